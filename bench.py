"""Benchmark of the fused SSD prefill forward: one JSON line on stdout.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one call of the whole fused path (chunk cumsum, BMM, chunk state,
state passing, chunk scan) over one batch of synthetic inputs. The default
workload is the long-context layer (batch 1, seqlen 262144, 80 heads in 8
groups, headdim 64, d_state 128, chunk 128, bf16 I/O, fp32 states, no initial
state), the largest of the single-GPU workloads: its 6.5 GB of inputs and
outputs are far larger than L2, and a 512 MiB buffer is still written before
every step, outside the timed events (other workloads fit in L2). The step
time is the median of the per-step CUDA-event timings.

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the (batch, head) chains need no exchange); the time is the
maximum over ranks and the value counts all ranks' tokens.

--impl reference times the CPU oracle (fp64 token-by-token recurrence) on the
host cores instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mamba_ssd_prefill_gb300.inputs import DTYPES, WORKLOADS, make_chain_inputs, make_inputs  # noqa: E402

METRIC = "SSD prefill tokens/s per layer at 1 GB300; % of roofline (HBM vs tensor)"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "long-L256k-g8"
FLUSH_BYTES = 512 * 1024 * 1024


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def algorithmic(w):
    """Algorithmic bytes and causal MMA flops of one call (on-chip intermediates not counted)."""
    T = w.batch * w.seqlen
    e = 4 if w.io == "f32" else 2
    es = 4 if w.state == "f32" else 2
    states = w.batch * w.nheads * w.headdim * w.dstate * es
    nbytes = T * e * (2 * w.nheads * w.headdim + w.nheads + 2 * w.ngroups * w.dstate)
    nbytes += states * (2 if w.init != "none" else 1)  # init read (when given) + final write
    q1 = (w.chunk + 1) / 2.0
    macs = T * (w.ngroups * w.dstate * q1 + w.nheads * w.headdim * q1 + 2 * w.nheads * w.dstate * w.headdim)
    return nbytes, 2.0 * macs


def kernel_hash():
    h = hashlib.sha256()
    for f in ("ssd_tc.cu", "sm100_ptx.cuh", "ssd_common.cuh"):  # the fused kernel's sources
        h.update(open(os.path.join(ROOT, "mamba_ssd_prefill_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples (every 20 ms, host-timestamped) while the GPU is under load."""

    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.rows = []
        self.window = None

    def __enter__(self):
        import threading

        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except OSError:
            self.proc = None
            return self
        self.started = threading.Event()

        def reader():
            for line in self.proc.stdout:
                self.rows.append((time.perf_counter(), line.strip()))
                self.started.set()

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        self.started.wait(timeout=5.0)  # sampler is running before the timed region starts
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0, t1, t_load_end):
        """Samples taken in [t0, t1] (the timed region); if none, those up to t_load_end (identical untimed steps
        run right after it), saying so."""
        def parse(lo, hi):
            out = []
            for ts, line in self.rows:
                if lo <= ts <= hi:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) == 6:
                        try:
                            out.append((float(parts[0]), float(parts[1]), parts[2:]))
                        except ValueError:
                            pass
            return out

        rows, where = parse(t0, t1), "timed region"
        if not rows:
            rows, where = parse(t0, t_load_end), "timed region and the identical untimed steps right after it"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "window": where}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, tokens_per_rank, ms_per_step_max):
    """Whole-job tokens/s of `world` independent replicas, timed by the slowest rank."""
    return world * tokens_per_rank / (ms_per_step_max * 1e-3)


def device_chains(w, inp, n, rng):
    """n random (sequence, head) chains of the device inputs, copied to the host as float64 (only those chains)."""
    b, L, H, P = inp["x"].shape
    per = H // w.ngroups
    order = [(bi, h) for bi in range(b) for h in range(H)]
    rng.shuffle(order)
    ch = order[:min(n, len(order))]
    hs = np.array([h for _, h in ch])

    def stack(f):
        return torch.stack([f(bi, h) for bi, h in ch]).double().cpu().numpy()

    init = None if inp["init_states"] is None else stack(lambda bi, h: inp["init_states"][bi, h])
    return dict(x=stack(lambda bi, h: inp["x"][bi, :, h]), dt_raw=stack(lambda bi, h: inp["dt_raw"][bi, :, h]),
                dt_bias=inp["dt_bias"].double().cpu().numpy()[hs], A=inp["A"].double().cpu().numpy()[hs],
                B=stack(lambda bi, h: inp["B"][bi, :, h // per]), C=stack(lambda bi, h: inp["C"][bi, :, h // per]),
                D=inp["D"].double().cpu().numpy()[hs], init=init), len(order)


def oracle_sample(w, chains, total_chains, budget_s, min_reps=1):
    """Time the oracle on whole chains (float64 arrays of a sample of the workload's chains) for about budget_s;
    returns (tokens/s, sample text, threads)."""
    import oracle

    threads = oracle.default_threads()
    n, L = chains["x"].shape[0], chains["x"].shape[1]
    args = (chains["x"], chains["dt_raw"], chains["dt_bias"], chains["A"], chains["B"], chains["C"], chains["D"],
            chains["init"])
    t0 = time.perf_counter()
    oracle.ssd_chains(*args, nthreads=threads)
    dt1 = time.perf_counter() - t0
    reps = max(min_reps, int(budget_s / max(dt1, 1e-3)))
    reps = min(reps, 50)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.ssd_chains(*args, nthreads=threads)
    el = time.perf_counter() - t0
    chain_tokens = reps * n * L
    tok_s = chain_tokens / w.nheads / el  # a token is one position across all heads
    sample = (f"{n} of {total_chains} (sequence, head) chains x {L} tokens, {reps} repetitions, "
              f"{el:.1f} s; tokens/s = chain-tokens / nheads / seconds")
    return tok_s, sample, threads


def run_reference(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle

    # only the sampled chains are drawn (the whole long-context batch would be gigabytes of host arrays)
    chains = make_chain_inputs(w, min(w.batch * w.nheads, oracle.default_threads()))
    cfg = workload_config(w)
    cfg["reference_inputs"] = "the sampled chains drawn directly with the workload's recipe (make_chain_inputs)"
    per_step = []
    budget = min(args.ref_budget, 150.0 / (args.warmup + args.steps))  # whole run within a few minutes
    for s in range(args.warmup + args.steps):
        tok_s, sample, threads = oracle_sample(w, chains, w.batch * w.nheads, budget_s=budget)
        if s >= args.warmup:
            per_step.append(tok_s)
    v = float(np.median(per_step))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": w.tokens / v * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w):
    return {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads, "headdim": w.headdim,
            "dstate": w.dstate, "ngroups": w.ngroups, "chunk": w.chunk, "io": w.io, "state": w.state,
            "init_states": w.init, "parallelism": "replicas"}


def run_gpu(args, w):
    import mamba_ssd_prefill_gb300 as m

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    if args.segment_chunks != -1:
        m.debug_knobs(tc_segment_chunks=args.segment_chunks)
    dev = torch.device("cuda", local)
    st = DTYPES[w.state]
    inp = make_inputs(w, device=dev, seed=w.seed + rank)
    prob = m.make_problem(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk, DTYPES[w.io], st)
    kernel = m.kernel_for(prob)
    plan = m.plan_info(prob)
    ws = m.Workspace(dev)
    y = torch.empty_like(inp["x"])
    fin = torch.empty(w.batch, w.nheads, w.headdim, w.dstate, dtype=st, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        m.ssd_fwd(**inp, chunk_size=w.chunk, state_dtype=st, workspace=ws, y=y, final_states=fin)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    m.check(ws)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()  # L2 flush, outside the events
            torch.cuda._sleep(400000)  # keeps the GPU busy while the host marshals the call: no host gap is timed
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        wall1 = time.perf_counter()
        wall = wall1 - wall0
        load_end = wall1
        while wall < 0.3 and time.perf_counter() - wall1 < 0.3:  # short region: keep the same load for the sampler
            for _ in range(10):
                flush.zero_()
                step()
            torch.cuda.synchronize(dev)
            load_end = time.perf_counter()
    barrier(world)
    m.check(ws)
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(float(np.median(times)), world)
    value = replica_throughput(world, w.tokens, ms)

    # end to end through the public API with host buffers: ssd_fwd_host takes the pinned host inputs and outputs
    # (the layer parameters dt_bias, A, D stay on the device) and streams the batch through the GPU in token pieces,
    # the H2D copy of one piece and the D2H copy of another overlapping the computation of a third
    params = {k: inp[k] for k in ("dt_bias", "A", "D")}
    host = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in inp.items() if k not in params}
    y_host = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    f_host = torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = y.numel() * y.element_size() + fin.numel() * fin.element_size()
    scratch = m.Workspace(dev)

    def e2e_step():
        m.ssd_fwd_host(**host, **params, chunk_size=w.chunk, state_dtype=st, y=y_host, final_states=f_host,
                       scratch=scratch, stream=stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    m.check(scratch)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)

    if rank != 0:
        return
    hbm, tflops, kind = peaks()
    nbytes, flops = algorithmic(w)
    achieved = nbytes / (ms * 1e-3) / 1e9
    t_mem, t_tc = nbytes / (hbm * 1e9), flops / (tflops * 1e12)
    bound = "hbm" if t_mem >= t_tc else "tensor"
    roof = {"bound": bound, "achieved": achieved if bound == "hbm" else flops / (ms * 1e-3) / 1e12,
            "peak": hbm if bound == "hbm" else tflops, "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "traffic": traffic_for(w.name), "peak_kind": kind,
            "roofline_time_us": max(t_mem, t_tc) * 1e6, "algorithmic_bytes": nbytes, "causal_flops": flops}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if bound == "hbm":  # beside the measured peak: the fraction of the nominal 7.9 TB/s of HBM3e (the stricter one)
        roof["frac_of_nominal_7900_gbs"] = achieved / NOMINAL_HBM_GBS
    cfg = workload_config(w)
    # the per-token dt the inputs realise (softplus of dt_raw + dt_bias), outside any timed region
    with torch.no_grad():
        dtv = torch.nn.functional.softplus(inp["dt_raw"].float() + inp["dt_bias"].float())
        cfg["dt_realised"] = [float(dtv.min()), float(dtv.max())]
        del dtv
    cfg.update({"kernel": kernel, "segments": plan["segments"], "segment_chunks": plan["segment_chunks"],
                "launches_per_step": plan["launches"],
                "state_flags": "one release flag per head" if plan["head_flags"] else "per state row (fp32) or tagged words (fp16)",
                "l2": f"{FLUSH_BYTES >> 20} MiB buffer written before every step, outside the events",
                "wall_s_timed_region": round(wall, 3)})
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic", "config": cfg, "roofline": roof,
            "e2e": {"value": world * w.tokens / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "path": "ssd_fwd_host: pinned host buffers streamed in token pieces of about 256 MiB of copies, 8 to 32 (copies overlap compute)"},
            "gpu_launches": args.steps * plan["launches"], "clocks": clk.summary(wall0, wall1, load_end)}
    if world == 1 and not args.no_cpu_baseline:
        import oracle

        chains, total = device_chains(w, inp, oracle.default_threads(), np.random.default_rng(0))
        tok_s, sample, threads = oracle_sample(w, chains, total, budget_s=args.ref_budget)
        line["cpu_baseline"] = {"value": tok_s, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-budget", type=float, default=12.0, help="seconds of oracle work per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--segment-chunks", type=int, default=-1,
                    help="two-level state passing: chunks per segment (0: one chain per sequence; default: the "
                         "library's choice); for profiling the segment kernels on reduced workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
