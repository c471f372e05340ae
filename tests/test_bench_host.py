"""bench.py's host-side arithmetic (no GPU): the roofline's algorithmic bytes and flops, the replica throughput,
the traffic record's source check and the clock record's throttle reasons."""
import bench
from mamba_ssd_prefill_gb300.inputs import WORKLOADS


def per_token(name):
    w = WORKLOADS[name]
    b, f = bench.algorithmic(w)
    T = w.batch * w.seqlen
    return b / T, f / T


def test_algorithmic_bytes_and_flops_per_token():
    """Per token: e·(2HP + H + 2GN) bytes of x, dt_raw, B, C and y, plus the [b, H, P, N] states (an initial state
    read when one is given, the final one written), and 2·(GN(Q+1)/2 + HP(Q+1)/2 + 2HNP) causal MMA flops. The
    values are worked out by hand from the layer shapes (tiny: H=8, P=N=64, fp32; 130M: H=24, P=64, N=128, bf16,
    4 x 4096 tokens, fp32 states; 2.7B: H=80)."""
    assert per_token("tiny-fp32") == (4 * (2 * 8 * 64 + 8 + 2 * 64) + 2 * 8 * 64 * 64 * 4 / 1024,
                                      2 * (64 * 64.5 + 512 * 64.5 + 2 * 8 * 64 * 64))
    b, f = per_token("m130-bf16")
    assert b == 7088.0 and f == 1001088.0  # 2 (3072 + 24 + 256) + 2 x 4 x 24 x 64 x 128 x 4 / 16384
    b, f = per_token("m2p7-L8k-b1")
    assert b == 21792.0 and f == 2 * (128 * 64.5 + 5120 * 64.5 + 2 * 80 * 128 * 64)
    b, _ = per_token("m2p7-L16k-q128")  # no initial state: only the fp16 final state is written
    assert b == 2 * (10240 + 80 + 256) + 80 * 64 * 128 * 2 / 16384
    _, f256 = per_token("m2p7-L16k-q256")
    assert f256 == 2 * (128 * 128.5 + 5120 * 128.5 + 2 * 80 * 128 * 64)


def test_replica_throughput_counts_every_rank():
    assert bench.replica_throughput(1, 16384, 0.1) == 16384 / 1e-4
    assert bench.replica_throughput(4, 16384, 0.2) == 4 * 16384 / 2e-4


def test_traffic_record_only_for_the_source_it_was_taken_on(monkeypatch):
    real = bench.traffic_for("m130-bf16")
    assert real is None or real > 0
    monkeypatch.setattr(bench, "kernel_hash", lambda: "0" * 16)
    assert bench.traffic_for("m130-bf16") is None
    assert bench.traffic_for("no-such-workload") is None


def test_clock_summary_reports_throttle_reasons_and_falls_back_to_the_steps_after():
    c = bench.ClockSampler(0)
    c.rows = [(1.0, "2070, 2070, Not Active, Not Active, Not Active, Not Active"),
              (1.5, "2055, 2070, Not Active, Not Active, Not Active, Active"),
              (2.0, "2070, 2070, Not Active, Not Active, Not Active, Not Active"),
              (3.5, "1800, 2070, Active, Not Active, Not Active, Not Active"),
              (3.6, "garbled")]
    s = c.summary(0.9, 2.1, 4.0)
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["window"] == "timed region"
    s = c.summary(2.5, 3.0, 4.0)  # nothing inside the timed region: the identical steps right after it
    assert s["samples"] == 1 and s["reasons"] == ["hw_slowdown"] and s["sm_mhz"] == 1800.0
    assert bench.ClockSampler(0).summary(0, 1, 2)["reasons"] == ["unsampled"]
