"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element."""
import math
import os

import numpy as np
import pytest
import torch

import mamba_ssd_prefill_gb300 as m
import oracle
from mamba_ssd_prefill_gb300.inputs import DTYPES, WORKLOADS, make_conv_inputs, make_inputs
from parity import gate_final, gate_y, gate_y_tc_envelope

pytestmark = pytest.mark.gpu



@pytest.fixture
def knobs():
    """Forces launch-configuration choices through the ssd_debug_knobs test hook; the library's own choices are
    restored afterwards."""
    state = {}

    def set_(**kw):
        state.update(kw)
        m.debug_knobs(**state)

    yield set_
    m.debug_knobs()

def cpu(d):
    return {k: (v.cpu() if v is not None else None) for k, v in d.items()}


def run_gpu(w, inp, kernel="auto", ws=None, **kw):
    ws = ws or m.Workspace("cuda")
    y, fin = m.ssd_fwd(**inp, chunk_size=w.chunk, state_dtype=DTYPES[w.state], kernel=kernel, workspace=ws, **kw)
    m.check(ws)
    return y, fin


def auto_kernel(w):
    """The kernel ssd_fwd picks for workload w under SSD_KERNEL_AUTO."""
    return m.kernel_for(m.make_problem(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk,
                                       DTYPES[w.io], DTYPES[w.state]))


def assert_parity(w, y, fin, yr, fr, label="", kernel=None):
    """y and the final states against the oracle; kernel: the kernel that ran ("auto" or None: ssd_fwd's choice)."""
    k = auto_kernel(w) if kernel in (None, "auto") else kernel
    ok, s = gate_y(y.double().cpu().numpy(), yr, w.io, w.state, tc=k == "tc")
    assert ok, f"{label} y parity failed: {s}"
    okf, sf = gate_final(fin.double().cpu().numpy(), fr, w.io, w.state)
    assert okf, f"{label} final-state parity failed: {sf}"
    return s


SMALL = [
    # (workload, overrides)
    ("tiny-fp32", {}),                                                               # the full tiny fp32 config
    ("tiny-fp32", dict(seqlen=300, chunk=64, nheads=3, ngroups=3, init="normal")),    # ragged tail, groups
    ("m130-bf16", dict(batch=2, seqlen=300, nheads=4, ngroups=2, chunk=64)),          # bf16, ragged, 2 groups
    ("m130-bf16", dict(batch=1, seqlen=257, nheads=2, chunk=256, io="f16", state="f16")),
    ("m130-bf16", dict(batch=3, seqlen=1, nheads=2, chunk=128)),                      # one token
    ("m130-bf16", dict(batch=1, seqlen=200, nheads=2, headdim=32, dstate=16, chunk=48)),  # other dims
]


@pytest.mark.parametrize("name,over", SMALL, ids=[f"{n}-{i}" for i, (n, _) in enumerate(SMALL)])
def test_simt_parity_small(name, over):
    w = WORKLOADS[name].with_(**over)
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp, kernel="simt")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, f"simt {name} {over}", kernel="simt")


@pytest.mark.parametrize("two_pass", ["0", "1"])
@pytest.mark.parametrize("name,over", [
    ("tiny-fp32", {}),
    ("m130-bf16", dict(batch=2, seqlen=300, nheads=3, ngroups=3, chunk=64, headdim=32, dstate=64, state="f16",
                       init="normal")),
    ("tiny-fp32", dict(batch=3, seqlen=200, nheads=2, chunk=32, init="normal")),
], ids=["tiny", "bf16-f16-ragged", "fp32-init"])
def test_simt_one_and_two_passes(name, over, two_pass, knobs):
    """The SIMT kernel walks each chunk once (the entering state awaited first) or twice (the chunk state from zero
    first, the leaving state published right after the wait, then y): both against the oracle."""
    knobs(simt_two_pass=int(two_pass))
    w = WORKLOADS[name].with_(**over)
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp, kernel="simt")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, f"simt two_pass={two_pass} {name} {over}", kernel="simt")


def test_simt_no_D_no_init():
    w = WORKLOADS["m130-bf16"].with_(batch=1, seqlen=150, nheads=2, init="none")
    inp = make_inputs(w, device="cuda")
    inp["D"] = None
    y, fin = run_gpu(w, inp, kernel="simt")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr)


def test_split_and_rerun_matches_full():
    """Resume semantics: [0, T1) then [T1, L) with init = the first part's final state."""
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=333, nheads=2, chunk=64)
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp, kernel="simt")
    for T1 in (64, 100):
        a = {k: v for k, v in inp.items()}
        b = {k: v for k, v in inp.items()}
        for k in ("x", "dt_raw", "B", "C"):
            a[k] = inp[k][:, :T1].contiguous()
            b[k] = inp[k][:, T1:].contiguous()
        y1, s1 = run_gpu(w, a, kernel="simt")
        b["init_states"] = s1
        y2, f2 = run_gpu(w, b, kernel="simt")
        yc = torch.cat([y1, y2], dim=1).double().cpu().numpy()
        ok, s = gate_y(yc, y.double().cpu().numpy(), w.io)
        assert ok, s
        assert np.max(np.abs(f2.double().cpu().numpy() - fin.double().cpu().numpy())) <= 1e-3


def test_deterministic_and_workspace_reuse():
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=400, nheads=3, chunk=128)
    inp = make_inputs(w, device="cuda")
    ws = m.Workspace("cuda")
    y1, f1 = run_gpu(w, inp, kernel="simt", ws=ws)
    for _ in range(3):
        y2, f2 = run_gpu(w, inp, kernel="simt", ws=ws)
        assert torch.equal(y1, y2) and torch.equal(f1, f2)


def test_final_states_may_alias_init():
    w = WORKLOADS["m130-bf16"].with_(batch=1, seqlen=300, nheads=2, chunk=128)
    inp = make_inputs(w, device="cuda")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    st = inp["init_states"]
    y, fin = run_gpu(w, inp, kernel="simt", final_states=st)
    assert fin.data_ptr() == st.data_ptr()
    assert_parity(w, y, fin, yr, fr)


def test_empty_sequence_copies_init():
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=0, nheads=2)
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp)
    assert y.numel() == 0
    assert torch.equal(fin, inp["init_states"])
    inp["init_states"] = None
    y, fin = run_gpu(w, inp)
    assert torch.count_nonzero(fin) == 0


def test_injected_missing_publish_times_out_and_recovers():
    """Host-armed fault injection: chunk 1's publish is skipped, chunk 2's wait runs
    out of time, the kernel returns with SSD_ERR_TIMEOUT; the workspace then works again."""
    w = WORKLOADS["m130-bf16"].with_(batch=1, seqlen=512, nheads=2, chunk=128)
    inp = make_inputs(w, device="cuda")
    ws = m.Workspace("cuda")
    y0, f0 = run_gpu(w, inp, kernel="simt", ws=ws)
    m.debug_set(ws, timeout_ns=50_000_000, skip_publish=1)
    m.ssd_fwd(**inp, chunk_size=w.chunk, kernel="simt", workspace=ws)
    with pytest.raises(m.SsdError) as e:
        m.check(ws)
    assert e.value.status == 5
    m.debug_set(ws, timeout_ns=0, skip_publish=-1)
    y1, f1 = run_gpu(w, inp, kernel="simt", ws=ws)
    assert torch.equal(y0, y1) and torch.equal(f0, f1)


# ----------------------------------------------------------------------------- tensor-core kernel
TC_SMALL = [
    ("m130-bf16", dict(batch=2, seqlen=300, nheads=4, ngroups=2)),              # ragged tail, 2 groups
    ("m130-bf16", dict(batch=1, seqlen=257, nheads=2, io="f16", state="f16")),  # fp16 I/O and states
    ("m130-bf16", dict(batch=3, seqlen=1, nheads=2)),                           # one token
    ("m130-bf16", dict(batch=1, seqlen=2048, nheads=8, init="none")),           # 16 chunks, no init
    ("m130-bf16", dict(batch=2, seqlen=1000, nheads=6, ngroups=3, state="f16")),
    ("m130-bf16", dict(batch=2, seqlen=700, nheads=4, chunk=256)),              # chunk 256, run as 128s
]


@pytest.mark.parametrize("name,over", TC_SMALL, ids=[f"{n}-{i}" for i, (n, _) in enumerate(TC_SMALL)])
def test_tc_parity_small(name, over):
    w = WORKLOADS[name].with_(**over)
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp, kernel="tc")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, f"tc {name} {over}", kernel="tc")


@pytest.mark.parametrize("dt_bias,A", [(-6.0, -0.5), (2.0, -16.0), (0.5, None)],
                         ids=["weak-decay", "strong-decay", "mixed-decay"])
def test_decay_regimes(dt_bias, A):
    """Decay from almost none to total within a few tokens, so both ways of forming the decay mask run:
    the two-factor split and the direct exponential of the diagonal blocks (decay range over 100 in log2).
    The strong and mixed cases drive |y| into the hundreds and the states far above 10, well outside the
    pages' workloads: there the SIMT kernel (fp32 throughout) still meets the gate, and the tensor-core
    kernel, whose P, X_s and S_in are fp16, is held to its operand envelope."""
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=777, nheads=6, ngroups=2, seed=77)
    inp = make_inputs(w, device="cuda")
    inp["dt_bias"] = torch.full_like(inp["dt_bias"], dt_bias)
    if A is None:  # per head from -16 to -0.01
        inp["A"] = -torch.logspace(math.log10(16.0), -2.0, w.nheads, device="cuda", dtype=torch.float32)
    else:
        inp["A"] = torch.full_like(inp["A"], A)
    yr, fr = oracle.ssd_reference(**cpu(inp))
    y, fin = run_gpu(w, inp, kernel="simt")
    assert_parity(w, y, fin, yr, fr, f"simt decay dt_bias={dt_bias} A={A}", kernel="simt")
    y, fin = run_gpu(w, inp, kernel="tc")
    if dt_bias < 0:  # inside the pages' regime: the plain gate
        assert_parity(w, y, fin, yr, fr, f"tc decay dt_bias={dt_bias} A={A}", kernel="tc")
    else:
        ok, s = gate_y_tc_envelope(y.double().cpu().numpy(), yr)
        assert ok, f"tc decay dt_bias={dt_bias} A={A}: {s}"


@pytest.mark.parametrize("hs", [1, 2, 4, 8])
def test_tc_heads_per_unit(hs, knobs):
    knobs(tc_heads_per_unit=hs)
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=700, nheads=16, ngroups=2, seed=50 + hs)
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp, kernel="tc")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, f"tc hs={hs}", kernel="tc")


@pytest.mark.parametrize("late", ["0", "1"], ids=["early-tickets", "late-tickets"])
@pytest.mark.parametrize("hs", [1, 2, 8])
def test_tc_ticket_order(late, hs, knobs):
    """Work units taken one unit ahead or only when the unit before nears its end (every head count, so the
    signal comes from the first, a middle and a late head of a unit): same results, and bit for bit the same."""
    knobs(tc_late_ticket=int(late), tc_heads_per_unit=hs)
    w = WORKLOADS["m130-bf16"].with_(batch=3, seqlen=1100, nheads=16, seed=70 + hs)
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp, kernel="tc")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, f"tc late={late} hs={hs}", kernel="tc")
    knobs(tc_late_ticket=1 if late == "0" else 0)
    y2, f2 = run_gpu(w, inp, kernel="tc")
    assert torch.equal(y, y2) and torch.equal(fin, f2)


SEGMENTS = [
    # (workload, overrides, chunks per segment): two-level state passing forced through the test hook
    ("m130-bf16", dict(batch=2, seqlen=2000, nheads=8, ngroups=2), 3),                 # 16 chunks: 6 segments, ragged
    ("m130-bf16", dict(batch=1, seqlen=4096, nheads=16, ngroups=2, io="f16", state="f16"), 8),
    ("m130-bf16", dict(batch=3, seqlen=1500, nheads=10, ngroups=2), 2),                # 5 heads per unit (odd)
    ("m130-bf16", dict(batch=2, seqlen=1024, nheads=4, state="f16"), 1),               # every chunk a segment
    ("long-L256k-g8", dict(seqlen=16384, nheads=16), 32),                              # 8 groups, fp32, no init
    ("m130-bf16", dict(batch=1, seqlen=3000, nheads=24, init="none", dt_lo=1e-4), 5),  # slow decay, no init
]


@pytest.mark.parametrize("name,over,seg", SEGMENTS, ids=[f"seg{i}" for i in range(len(SEGMENTS))])
def test_tc_segmented_state_passing(name, over, seg, knobs):
    """Two-level state passing: block aggregates and segment entering states computed before the fused kernel,
    whose state chain then restarts at every segment start. Against the oracle, and against the one-chain run."""
    w = WORKLOADS[name].with_(**over)
    inp = make_inputs(w, device="cuda")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    knobs(tc_segment_chunks=seg)
    y, fin = run_gpu(w, inp, kernel="tc")
    assert_parity(w, y, fin, yr, fr, f"tc segments of {seg} {name} {over}", kernel="tc")
    knobs(tc_segment_chunks=0)
    y1, f1 = run_gpu(w, inp, kernel="tc")
    d = (y.double() - y1.double()).abs().max().item()
    assert d <= 1e-2 + 2e-2 * y1.double().abs().max().item(), d


@pytest.mark.parametrize("late", [0, 1], ids=["early-tickets", "late-tickets"])
@pytest.mark.parametrize("hs", [1, 4])
def test_tc_segments_with_tickets_and_heads(late, hs, knobs):
    """Segments together with every ticket order and head count: bit for bit the same across ticket orders."""
    knobs(tc_segment_chunks=4, tc_late_ticket=late, tc_heads_per_unit=hs)
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=2600, nheads=8, seed=90 + hs)
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp, kernel="tc")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, f"tc segments late={late} hs={hs}", kernel="tc")
    knobs(tc_late_ticket=1 - late)
    y2, f2 = run_gpu(w, inp, kernel="tc")
    assert torch.equal(y, y2) and torch.equal(fin, f2)


PLANS = [
    # workload: (segments, chunks per segment, per-head flags, launches) the library plans on a 152-SM GB300
    ("m130-bf16", (1, 32, False, 1)),
    ("m130-bf16-f16", (1, 32, False, 1)),
    ("m2p7-L16k-q128", (8, 16, True, 3)),
    ("m2p7-L8k-b1", (4, 16, False, 3)),
    ("m2p7-L8k-b8", (1, 64, True, 1)),
    ("m2p7-L8k-b8-f16", (1, 64, True, 1)),
    ("m2p7-L8k-b32", (1, 64, True, 1)),
    ("long-L256k-g8", (4, 512, False, 3)),
    ("long-L256k-g8-f16", (8, 256, True, 3)),
]


@pytest.mark.parametrize("name,want", PLANS, ids=[n for n, _ in PLANS])
def test_plans_of_the_measured_layers(name, want):
    """The launch plan of every measured layer on this GPU: two-level state passing where the chain outweighs
    the cadence (segments and their length), per-head state flags where many chains share a chunk position, and
    the launches a call makes. Pins the planning constants against the shapes they were measured on."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("plans measured on a 152-SM GB300")
    w = WORKLOADS[name]
    p = m.make_problem(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk, DTYPES[w.io],
                       DTYPES[w.state])
    info = m.plan_info(p)
    assert (info["segments"], info["segment_chunks"], info["head_flags"], info["launches"]) == want, info


@pytest.mark.parametrize("state", ["f32", "f16"])
@pytest.mark.parametrize("late", [0, 1], ids=["early-tickets", "late-tickets"])
@pytest.mark.parametrize("seg", [0, 4], ids=["one-chain", "segments"])
def test_tc_head_flags(state, late, seg, knobs):
    """States published behind one release flag per head (stored by the C.S warp once every row is written; fp16
    states then as plain halves) or the default way (fp32: a flag per row, by each row's thread; fp16: tagged
    words): the oracle's values, and the same bits either way, under both ticket orders, with and without
    segments."""
    w = WORKLOADS["m130-bf16"].with_(batch=3, seqlen=2200, nheads=8, ngroups=2, seed=97, state=state)
    inp = make_inputs(w, device="cuda")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    knobs(tc_late_ticket=late, tc_segment_chunks=seg, tc_head_flags=1)
    y, fin = run_gpu(w, inp, kernel="tc")
    assert_parity(w, y, fin, yr, fr, f"tc head flags {state} late={late} seg={seg}", kernel="tc")
    knobs(tc_head_flags=0)
    y2, f2 = run_gpu(w, inp, kernel="tc")
    assert torch.equal(y, y2) and torch.equal(fin, f2)


@pytest.mark.parametrize("fuse", [True, False], ids=["fused-conv", "conv-then-ssd"])
def test_tc_segments_repeat_and_conv_paths(fuse, knobs):
    """Repeated segmented launches on one workspace are bit-identical. With the convolution in front, the unfused
    path (convolved rows written first) runs segmented and the fused path (raw rows convolved as they load) keeps
    one chain per sequence under the same setting; both match the oracle."""
    knobs(tc_segment_chunks=2)
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=1300, nheads=8, ngroups=2)
    inp = make_inputs(w, device="cuda")
    ws = m.Workspace("cuda")
    y0, f0 = run_gpu(w, inp, kernel="tc", ws=ws)
    for _ in range(2):
        y1, f1 = run_gpu(w, inp, kernel="tc", ws=ws)
        assert torch.equal(y0, y1) and torch.equal(f0, f1)
    ci = make_conv_inputs(w, 4, device="cuda", seed=62)
    y, fin, cs, xo = m.ssd_fwd_conv(**ci, nheads=w.nheads, headdim=w.headdim, ngroups=w.ngroups, dstate=w.dstate,
                                    activation="silu", chunk_size=w.chunk, state_dtype=DTYPES[w.state], kernel="tc",
                                    workspace=ws, fuse=fuse)
    m.check(ws)
    assert (xo is None) == fuse
    yr, fr, _ = conv_reference(w, ci, 4, "silu")
    assert_parity(w, y, fin, yr, fr, f"conv fuse={fuse} with segments set", kernel="tc")


def test_tc_no_D_alias_and_determinism():
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=600, nheads=8)
    inp = make_inputs(w, device="cuda")
    inp["D"] = None
    yr, fr = oracle.ssd_reference(**cpu(inp))
    ws = m.Workspace("cuda")
    init = inp["init_states"].clone()
    y, fin = run_gpu(w, dict(inp, init_states=init), kernel="tc", ws=ws, final_states=init)
    assert fin.data_ptr() == init.data_ptr()
    assert_parity(w, y, fin, yr, fr)
    for _ in range(2):
        y2, f2 = run_gpu(w, inp, kernel="tc", ws=ws)
        assert torch.equal(y, y2) and torch.equal(fin, f2)


@pytest.mark.parametrize("state", ["f32", "f16"])  # flagged rows / tagged rows
def test_tc_injected_missing_publish_times_out_and_recovers(state):
    w = WORKLOADS["m130-bf16"].with_(batch=1, seqlen=1024, nheads=8, state=state)
    inp = make_inputs(w, device="cuda")
    ws = m.Workspace("cuda")
    y0, f0 = run_gpu(w, inp, kernel="tc", ws=ws)
    m.debug_set(ws, timeout_ns=50_000_000, skip_publish=2)
    m.ssd_fwd(**inp, chunk_size=w.chunk, state_dtype=DTYPES[w.state], kernel="tc", workspace=ws)
    with pytest.raises(m.SsdError) as e:
        m.check(ws)
    assert e.value.status == 5
    m.debug_set(ws, timeout_ns=0, skip_publish=-1)
    y1, f1 = run_gpu(w, inp, kernel="tc", ws=ws)
    assert torch.equal(y0, y1) and torch.equal(f0, f1)


def test_tc_matches_simt_kernel():
    """Both kernels against each other on the same inputs (a second, oracle-free cross-check)."""
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=900, nheads=8)
    inp = make_inputs(w, device="cuda")
    yt, ft = run_gpu(w, inp, kernel="tc")
    ys, fs = run_gpu(w, inp, kernel="simt")
    a, b = yt.double().cpu().numpy(), ys.double().cpu().numpy()
    # each output is within 1e-2 + 2^-8 |y| of the exact value, so the two are within twice that
    excess = np.abs(a - b) - (2e-2 + 2.0 ** -7 * np.abs(b))
    assert excess.max() <= 0, float(excess.max())


# full-size workloads, in the launch configuration the benchmark times; the oracle checks sampled chains
FULL = ["m130-bf16", "m2p7-L16k-q128", "m2p7-L16k-q256", "m2p7-L8k-b1", "m2p7-L8k-b8", "m2p7-L8k-b32",
        "long-L256k-g8", "m130-bf16-f16", "long-L256k-g8-f16"]


def sampled_chains(w, n):
    """n (batch, head) chains drawn at random, plus the first and the last chain and one random head of every group
    (in a random sequence), so that no group's B/C columns and no end of the chunk-major ticket order go unchecked."""
    g = np.random.default_rng(w.seed)
    all_c = [(b, h) for b in range(w.batch) for h in range(w.nheads)]
    if len(all_c) <= n:
        return all_c
    idx = sorted(g.choice(len(all_c), size=n, replace=False))
    per = w.nheads // w.ngroups
    groups = [(int(g.integers(w.batch)), gg * per + int(g.integers(per))) for gg in range(w.ngroups)]
    return sorted(set([all_c[0], all_c[-1]] + groups + [all_c[i] for i in idx]))


@pytest.mark.parametrize("name", FULL)
def test_tc_full_size_sampled(name, record_property):
    w = WORKLOADS[name]
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp)
    assert m.kernel_for(m.make_problem(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk,
                                       DTYPES[w.io], DTYPES[w.state])) == "tc"
    n = 96 if w.seqlen <= 4096 else (24 if w.seqlen <= 16384 else 16)
    chains = sampled_chains(w, n)
    per = w.nheads // w.ngroups
    sub = dict(
        x=torch.stack([inp["x"][b, :, h] for b, h in chains])[:, :, None].cpu(),
        dt_raw=torch.stack([inp["dt_raw"][b, :, h] for b, h in chains])[:, :, None].cpu(),
        B=torch.stack([inp["B"][b, :, h // per] for b, h in chains])[:, :, None].cpu(),
        C=torch.stack([inp["C"][b, :, h // per] for b, h in chains])[:, :, None].cpu(),
    )
    ys = torch.stack([y[b, :, h] for b, h in chains]).double().cpu().numpy()
    fs = torch.stack([fin[b, h] for b, h in chains]).double().cpu().numpy()
    hs = np.array([h for _, h in chains])
    init = None if inp["init_states"] is None else torch.stack([inp["init_states"][b, h] for b, h in chains])
    yr, fr = oracle.ssd_chains(sub["x"][:, :, 0], sub["dt_raw"][:, :, 0], inp["dt_bias"].cpu()[hs],
                               inp["A"].cpu()[hs], sub["B"][:, :, 0], sub["C"][:, :, 0], inp["D"].cpu()[hs],
                               None if init is None else init.cpu())
    ok, s = gate_y(ys, yr, w.io, w.state, tc=True)
    # the headroom under the gate (negative: every sampled element inside it), shown with pytest -rP
    print(f"PARITY {name}: {len(chains)} chains, y worst_margin {s['worst_margin']:.3e} (plain rule "
          f"{s['plain_worst_margin']:.3e}, {s['plain_ok']:.7f} of elements inside it), max|d| {s['max_abs']:.3e}, "
          f"match 1e-2 {s['match_1e-2']:.6f}")
    record_property("worst_margin", s["worst_margin"])
    assert ok, f"{name}: {s}"
    okf, sf = gate_final(fs, fr, w.io, w.state)
    assert okf, f"{name} final: {sf}"


# ----------------------------------------------------------------------------- single-token step (decode)
STEP = [
    ("m130-bf16", dict(batch=5, nheads=6, ngroups=2)),                                  # bf16, fp32 states
    ("m130-bf16", dict(batch=3, nheads=4, io="f16", state="f16")),                     # 16-byte fp16 vectors
    ("tiny-fp32", dict(batch=2, nheads=3, ngroups=3, init="normal")),                  # fp32, N = 64
    ("m130-bf16", dict(batch=2, nheads=2, headdim=24, dstate=100)),                    # N % 4 != 0: element-wise
    ("m130-bf16", dict(batch=64, nheads=80, init="none")),                             # no cached state yet
    ("m130-bf16", dict(batch=3, nheads=4, dstate=32)),                                 # 128-byte fp32 rows
    ("m130-bf16", dict(batch=2, nheads=4, dstate=64, state="f16")),                    # 128-byte fp16 rows
    ("m130-bf16", dict(batch=700, nheads=5, headdim=32, dstate=64, ngroups=5)),        # many chains per CTA
]


@pytest.mark.parametrize("name,over", STEP, ids=[f"{n}-{i}" for i, (n, _) in enumerate(STEP)])
def test_step_parity(name, over):
    w = WORKLOADS[name].with_(seqlen=1, **over)
    inp = make_inputs(w, device="cuda")
    assert m.kernel_for(m.make_problem(w.batch, 1, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk,
                                       DTYPES[w.io], DTYPES[w.state])) == "step"
    y, fin = run_gpu(w, inp)
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, f"step {name} {over}")


def test_step_in_place_without_D():
    w = WORKLOADS["m130-bf16"].with_(batch=4, seqlen=1, nheads=8)
    inp = make_inputs(w, device="cuda")
    inp["D"] = None
    yr, fr = oracle.ssd_reference(**cpu(inp))
    state = inp["init_states"].clone()
    y, fin = run_gpu(w, dict(inp, init_states=state), final_states=state)
    assert fin.data_ptr() == state.data_ptr()
    assert_parity(w, y, fin, yr, fr)


@pytest.mark.parametrize("state", ["f32", "f16"])
def test_step_without_final_states(state):
    """A step that returns y only (no state written) gives the same y as one that also writes the state."""
    w = WORKLOADS["m130-bf16"].with_(batch=9, seqlen=1, nheads=8, state=state, seed=95)
    inp = make_inputs(w, device="cuda")
    y_full, _ = run_gpu(w, inp)
    y_only, fin = run_gpu(w, inp, return_final_states=False)
    assert fin is None and torch.equal(y_only, y_full)


@pytest.mark.parametrize("state", ["f32", "f16"])
def test_decode_loop_matches_prefill(state):
    """Prefill a prompt with the tensor-core kernel, then decode six tokens one step at a time, the cached
    state updated in place: every step's y and the last state match the oracle over the whole sequence."""
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=300 + 6, nheads=4, state=state, seed=91)
    inp = make_inputs(w, device="cuda")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    T0 = 300
    pre = dict(inp, **{k: inp[k][:, :T0].contiguous() for k in ("x", "dt_raw", "B", "C")})
    y0, cache = run_gpu(w.with_(seqlen=T0), pre)
    ys = [y0]
    for t in range(T0, w.seqlen):
        tok = dict(inp, init_states=cache, **{k: inp[k][:, t:t + 1].contiguous() for k in ("x", "dt_raw", "B", "C")})
        yt, cache = run_gpu(w.with_(seqlen=1), tok, final_states=cache)
        ys.append(yt)
    y = torch.cat(ys, dim=1)
    assert_parity(w, y, cache, yr, fr, f"decode loop {state}")


@pytest.mark.parametrize("name", ["decode-2p7-b64", "decode-2p7-b256-f16"])
def test_step_full_size(name):
    w = WORKLOADS[name]
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp)
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, name)


@pytest.mark.parametrize("kernel,over", [("tc", {}), ("simt", {}), ("simt", dict(io="f32", state="f32")),
                                         ("step", dict(seqlen=1))],
                         ids=["tc", "simt-bf16", "simt-fp32", "step"])
def test_linear_attention_A_zero(kernel, over):
    """A = 0: no decay, the state is the running sum of dt x B^T (linear attention). Every kernel runs it with the
    same code; the oracle's A = 0 result is pinned to that closed form on the CPU."""
    w = WORKLOADS["m130-bf16"].with_(**dict(dict(batch=2, seqlen=400, nheads=4, ngroups=2, seed=31), **over))
    inp = make_inputs(w, device="cuda")
    inp["A"] = torch.zeros_like(inp["A"])
    # dt ~ 0.007: without decay the state is a growing sum; this keeps |y| in the pages' range (below ~20)
    inp["dt_bias"] = torch.full_like(inp["dt_bias"], -5.0)
    y, fin = run_gpu(w, inp, kernel=kernel)
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, f"A=0 {kernel}", kernel=kernel)


# ----------------------------------------------------------------------------- variable-length batches
from mamba_ssd_prefill_gb300.inputs import make_varlen_inputs  # noqa: E402

VARLEN = [
    ("tc", "m130-bf16", dict(nheads=4, ngroups=2), [300, 0, 1, 127, 128, 129, 700]),
    ("tc", "m130-bf16", dict(nheads=6, io="f16", state="f16", init="none"), [1000, 5, 256]),
    ("tc", "m130-bf16", dict(nheads=8), [0, 0, 64]),
    ("simt", "m130-bf16", dict(nheads=3, ngroups=3, chunk=64), [200, 0, 65, 1]),
    ("simt", "tiny-fp32", dict(nheads=2, init="normal"), [130, 7, 300]),
]


@pytest.mark.parametrize("kernel,name,over,lengths", VARLEN, ids=[f"{k}-{i}" for i, (k, *_r) in enumerate(VARLEN)])
def test_varlen_parity(kernel, name, over, lengths):
    w = WORKLOADS[name].with_(**over)
    inp = make_varlen_inputs(w, lengths, device="cuda", seed=101)
    ws = m.Workspace("cuda")
    y, fin = m.ssd_fwd_varlen(**inp, chunk_size=w.chunk, state_dtype=DTYPES[w.state], kernel=kernel, workspace=ws)
    m.check(ws)
    yr, fr = oracle.ssd_varlen_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, f"varlen {kernel} {lengths}", kernel=kernel)


def test_varlen_uniform_lengths_equal_regular_batch():
    w = WORKLOADS["m130-bf16"].with_(batch=3, seqlen=333, nheads=8)
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp)
    T = w.batch * w.seqlen
    packed = {k: (v.reshape(1, T, *v.shape[2:]) if k in ("x", "dt_raw", "B", "C") else v) for k, v in inp.items()}
    cu = torch.arange(0, T + 1, w.seqlen, dtype=torch.int32, device="cuda")
    yv, fv = m.ssd_fwd_varlen(**packed, cu_seqlens=cu, chunk_size=w.chunk, state_dtype=DTYPES[w.state])
    assert torch.equal(yv.reshape(y.shape), y) and torch.equal(fv, fin)


def test_varlen_bad_offsets_reported_then_recovers():
    w = WORKLOADS["m130-bf16"].with_(nheads=4)
    inp = make_varlen_inputs(w, [100, 50], device="cuda")
    ws = m.Workspace("cuda")
    good = inp["cu_seqlens"].clone()
    inp["cu_seqlens"] = torch.tensor([0, 120, 100], dtype=torch.int32, device="cuda")  # decreasing, wrong end
    m.ssd_fwd_varlen(**inp, chunk_size=w.chunk, workspace=ws)
    with pytest.raises(m.SsdError) as e:
        m.check(ws)
    assert e.value.status == 1
    inp["cu_seqlens"] = good
    y, fin = m.ssd_fwd_varlen(**inp, chunk_size=w.chunk, workspace=ws)
    m.check(ws)
    yr, fr = oracle.ssd_varlen_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr)


# ----------------------------------------------------------------------------- depthwise convolution in front
from mamba_ssd_prefill_gb300.inputs import make_conv_inputs  # noqa: E402

CONV = [
    ("tc", "m130-bf16", dict(batch=2, seqlen=333, nheads=4, ngroups=2), 4, "silu", True),   # fused, ragged, 2 seqs
    ("tc", "m130-bf16", dict(batch=2, seqlen=333, nheads=4, ngroups=2), 4, "silu", False),  # the same, unfused
    ("tc", "m130-bf16", dict(batch=3, seqlen=260, nheads=8, io="f16", state="f16"), 4, "none", True),
    ("tc", "m130-bf16", dict(batch=1, seqlen=700, nheads=8, io="f16", state="f16", init="none"), 3, "none", True),
    ("simt", "tiny-fp32", dict(batch=2, seqlen=200, nheads=2, init="normal"), 4, "silu", True),
    ("auto", "m130-bf16", dict(batch=3, seqlen=1, nheads=4), 4, "silu", True),               # decode step, cache
]


def conv_reference(w, inp, width, act):
    return oracle.ssd_conv_reference(inp["xbc"].cpu(), inp["conv_weight"].cpu(), inp["conv_bias"].cpu(),
                                     inp["dt_raw"].cpu(), inp["dt_bias"].cpu(), inp["A"].cpu(), w.nheads, w.headdim,
                                     w.ngroups, w.dstate, inp["D"].cpu(),
                                     None if inp["init_states"] is None else inp["init_states"].cpu(),
                                     None if inp["conv_state"] is None else inp["conv_state"].cpu(), act)


@pytest.mark.parametrize("kernel,name,over,width,act,fuse", CONV, ids=[f"{c[0]}-{i}" for i, c in enumerate(CONV)])
def test_conv_then_ssd_parity(kernel, name, over, width, act, fuse):
    w = WORKLOADS[name].with_(**over)
    inp = make_conv_inputs(w, width, device="cuda", seed=61, conv_state=w.batch != 3)
    ws = m.Workspace("cuda")
    y, fin, cs, xo = m.ssd_fwd_conv(**inp, nheads=w.nheads, headdim=w.headdim, ngroups=w.ngroups, dstate=w.dstate,
                                    activation=act, chunk_size=w.chunk, state_dtype=DTYPES[w.state], kernel=kernel,
                                    workspace=ws, fuse=fuse)
    m.check(ws)
    # fused exactly where the tensor-core kernel runs with width 4 (no activation buffer then)
    assert (xo is None) == (fuse and width == 4 and kernel == "tc")
    yr, fr, csr = conv_reference(w, inp, width, act)
    assert_parity(w, y, fin, yr, fr, f"conv {kernel} {over} fuse={fuse}", kernel=kernel)
    assert np.array_equal(cs.double().cpu().numpy(), csr)  # the cache holds the raw inputs exactly
    if xo is not None:
        xr, _ = oracle.conv1d_reference(inp["xbc"].cpu(), inp["conv_weight"].cpu(), inp["conv_bias"].cpu(),
                                        None if inp["conv_state"] is None else inp["conv_state"].cpu(), act)
        ok, s = gate_y(xo.double().cpu().numpy(), xr, w.io)  # the convolved rows, rounded once to the I/O dtype
        assert ok, s


@pytest.mark.parametrize("io,width,act", [("bf16", 4, "silu"), ("f16", 7, "none"), ("f32", 3, "silu")])
def test_conv_copy_pipeline_matches_tma_pipeline(io, width, act, knobs):
    """The conv kernel's two tile pipelines (one TMA box per tile, or 16-byte asynchronous copies, the form for rows
    that are not 16-byte multiples) convolve the same staged rows with the same arithmetic: bit-identical outputs
    and caches, and the oracle's values (ragged tiles: 333 tokens, a cache on entry)."""
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=333, nheads=4, ngroups=2, io=io, seed=64,
                                     **({"state": "f32", "chunk": 64} if io == "f32" else {}))
    inp = make_conv_inputs(w, width, device="cuda")
    kw = dict(nheads=w.nheads, headdim=w.headdim, ngroups=w.ngroups, dstate=w.dstate, activation=act,
              chunk_size=w.chunk, state_dtype=DTYPES[w.state])
    outs = []
    for tma in ("1", "0"):
        knobs(conv_tma=int(tma))
        ws = m.Workspace("cuda")
        outs.append(m.ssd_fwd_conv(**inp, **kw, workspace=ws, fuse=False))
        m.check(ws)
    (y1, f1, c1, x1), (y0, f0, c0, x0) = outs
    assert torch.equal(x1, x0) and torch.equal(c1, c0) and torch.equal(y1, y0) and torch.equal(f1, f0)
    xr, _ = oracle.conv1d_reference(inp["xbc"].cpu(), inp["conv_weight"].cpu(), inp["conv_bias"].cpu(),
                                    inp["conv_state"].cpu(), act)
    ok, s = gate_y(x0.double().cpu().numpy(), xr, w.io)
    assert ok, s


def test_conv_prefill_then_decode_continues_both_caches():
    """Prefill 250 tokens, then 3 single-token steps carrying the SSD state and the conv cache in place: every y and
    both final caches match the oracle over the whole 253-token sequence."""
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=253, nheads=4, seed=63)
    inp = make_conv_inputs(w, 4, device="cuda")
    yr, fr, csr = conv_reference(w, inp, 4, "silu")
    T0 = 250
    kw = dict(nheads=w.nheads, headdim=w.headdim, ngroups=w.ngroups, dstate=w.dstate, chunk_size=w.chunk)
    part = lambda a, b: {k: (v[:, a:b].contiguous() if k in ("xbc", "dt_raw") else v) for k, v in inp.items()}
    y0, state, cache, _ = m.ssd_fwd_conv(**part(0, T0), **kw)
    ys = [y0]
    for t in range(T0, w.seqlen):
        tok = part(t, t + 1)
        tok["init_states"], tok["conv_state"] = state, cache
        yt, state, cache, _ = m.ssd_fwd_conv(**tok, **kw, final_states=state, conv_state_out=cache)
        ys.append(yt)
    assert_parity(w, torch.cat(ys, dim=1), state, yr, fr, "conv prefill + decode")
    assert np.array_equal(cache.double().cpu().numpy(), csr)


# ----------------------------------------------------------------------------- CUDA graphs
def test_cuda_graph_prefill_and_decode_loop():
    """A prefill call and a loop of eight decode steps (state updated in place) are each captured once in a CUDA
    graph and replayed: the launches only read their workspace's epoch on the device, so replays need no host
    work, and they match eager execution bit for bit and the oracle over the whole sequence."""
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=264, nheads=8, seed=97)
    inp = make_inputs(w, device="cuda")
    yr, fr = oracle.ssd_reference(**cpu(inp))
    T0, steps = 256, 8
    pre = dict(inp, **{k: inp[k][:, :T0].contiguous() for k in ("x", "dt_raw", "B", "C")})
    toks = [dict(inp, **{k: inp[k][:, t:t + 1].contiguous() for k in ("x", "dt_raw", "B", "C")})
            for t in range(T0, T0 + steps)]
    wp, wd = w.with_(seqlen=T0), w.with_(seqlen=1)
    # eager reference run
    y_e, st_e = run_gpu(wp, pre)
    ys_e = []
    for tok in toks:
        yt, st_e = run_gpu(wd, dict(tok, init_states=st_e), final_states=st_e)
        ys_e.append(yt)
    # captured: workspaces and outputs allocated (and the library loaded) before capture
    ws_p, ws_d = m.Workspace("cuda"), m.Workspace("cuda")
    ws_p.get(m.workspace_size(m.make_problem(2, T0, 8, 64, 128, 1, 128)))
    ws_d.get(m.workspace_size(m.make_problem(2, 1, 8, 64, 128, 1, 128)))
    y_g = torch.empty_like(pre["x"])
    st_g = torch.empty_like(st_e)
    ys_g = [torch.empty_like(t["x"]) for t in toks]
    m.ssd_fwd(**pre, workspace=ws_p, y=y_g, final_states=st_g)  # warm-up outside the capture
    torch.cuda.synchronize()
    g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1):
        m.ssd_fwd(**pre, workspace=ws_p, y=y_g, final_states=st_g)
    with torch.cuda.graph(g2):
        for tok, yo in zip(toks, ys_g):
            m.ssd_fwd(**dict(tok, init_states=st_g), workspace=ws_d, y=yo, final_states=st_g)
    for _ in range(2):  # replays are repeatable: the prefill rewrites the state the decode loop advances
        g1.replay()
        g2.replay()
        torch.cuda.synchronize()
        m.check(ws_p)
        m.check(ws_d)
        assert torch.equal(y_g, y_e) and torch.equal(st_g, st_e)
        assert all(torch.equal(a, b) for a, b in zip(ys_g, ys_e))
    assert_parity(w, torch.cat([y_g] + ys_g, dim=1), st_g, yr, fr, "graph replay")


# ----------------------------------------------------------------------------- host-resident batches
def _pinned(t):
    return None if t is None else t.cpu().pin_memory()


@pytest.mark.parametrize("case", ["batch-5", "one-sequence", "f16-states", "simt-fp32", "pageable"])
def test_host_streaming_matches_device_call(case):
    """ssd_fwd_host streams host tensors through the GPU in token pieces of the whole batch, the states running
    from piece to piece: the same chunks in the same order and precision as one device call, so y and the final
    states are bit for bit those of ssd_fwd, and within the parity gate of the oracle."""
    over = {"batch-5": dict(batch=5, seqlen=700, nheads=8),
            "one-sequence": dict(batch=1, seqlen=1100, nheads=8),
            "f16-states": dict(batch=2, seqlen=1000, nheads=6, state="f16"),
            "simt-fp32": dict(batch=2, seqlen=900, nheads=4, io="f32", chunk=64),
            "pageable": dict(batch=3, seqlen=300, nheads=4)}[case]
    w = WORKLOADS["m130-bf16"].with_(seed=300 + len(case), **over)
    inp = make_inputs(w, device="cuda")
    st = DTYPES[w.state]
    y_d, f_d = m.ssd_fwd(**inp, chunk_size=w.chunk, state_dtype=st)
    host = {k: (v if k in ("dt_bias", "A", "D") else (v.cpu() if case == "pageable" else _pinned(v)))
            for k, v in inp.items()}
    scratch = m.Workspace("cuda")
    y_h, f_h = m.ssd_fwd_host(**host, chunk_size=w.chunk, state_dtype=st, pieces=3 if case == "one-sequence" else 0,
                              scratch=scratch)
    torch.cuda.synchronize()
    m.check(scratch)
    assert torch.equal(y_h, y_d.cpu()) and torch.equal(f_h, f_d.cpu())
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y_h, f_h, yr, fr, f"host {case}")


def test_host_streaming_piece_counts_and_empty():
    """Every piece count from one to more pieces than there are chunks gives the same result; a sequence of
    length 0 returns the initial states as the final ones."""
    w = WORKLOADS["m130-bf16"].with_(batch=1, seqlen=520, nheads=4, seed=333)
    inp = make_inputs(w, device="cuda")
    host = {k: (v if k in ("dt_bias", "A", "D") else _pinned(v)) for k, v in inp.items()}
    y_d, f_d = m.ssd_fwd(**inp, chunk_size=w.chunk)
    scratch = m.Workspace("cuda")
    for pieces in (1, 2, 4, 5, 9):
        y_h, f_h = m.ssd_fwd_host(**host, chunk_size=w.chunk, pieces=pieces, scratch=scratch)
        torch.cuda.synchronize()
        assert torch.equal(y_h, y_d.cpu()) and torch.equal(f_h, f_d.cpu()), pieces
    # from 8 pieces on, short first and last pieces (33 chunks, the last ragged: 1, 5, ..., 5, 2 or 1, 3, ..., 1)
    w2 = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=4100, nheads=4, seed=335)
    inp2 = make_inputs(w2, device="cuda")
    host2 = {k: (v if k in ("dt_bias", "A", "D") else _pinned(v)) for k, v in inp2.items()}
    y_d2, f_d2 = m.ssd_fwd(**inp2, chunk_size=w2.chunk)
    for pieces in (0, 8, 12):
        y_h, f_h = m.ssd_fwd_host(**host2, chunk_size=w2.chunk, pieces=pieces, scratch=scratch)
        torch.cuda.synchronize()
        assert torch.equal(y_h, y_d2.cpu()) and torch.equal(f_h, f_d2.cpu()), pieces
    e = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=0, nheads=4, seed=334)
    ie = make_inputs(e, device="cuda")
    he = {k: (v if k in ("dt_bias", "A", "D") else _pinned(v)) for k, v in ie.items()}
    y0, f0 = m.ssd_fwd_host(**he, chunk_size=e.chunk, scratch=scratch)
    torch.cuda.synchronize()
    assert y0.numel() == 0 and torch.equal(f0, he["init_states"])


# ----------------------------------------------------------------------------- bounds-checked debug build
def test_bounds_checked_build_reports_no_violation_and_catches_the_probe():
    """The debug build compares every kernel's global indices with the buffers' extents (an index outside is never
    used and is reported). Every entry point on edge-case shapes runs clean under it; the planted probe (the
    tensor-core kernel's dt_raw indices one extent too far) is caught and reported, and the workspace works again
    after it."""
    import subprocess
    import sys

    from mamba_ssd_prefill_gb300 import _build

    lib_path = _build.build(checked=True)
    env = dict(os.environ, MAMBA_SSD_LIB=lib_path)
    r = subprocess.run([sys.executable, os.path.join(os.path.dirname(__file__), "bounds_cases.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    results = dict(line.split() for line in r.stdout.strip().splitlines())
    assert len(results) == 16, results
    assert results.pop("probe") == "6", r.stdout
    assert all(v == "0" for v in results.values()), results


def test_host_streaming_in_a_cuda_graph():
    """ssd_fwd_host captured once in a CUDA graph (its copy streams join the capture through the events on the
    caller's stream) and replayed: the replays give the same y and final states as the eager call."""
    w = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=520, nheads=4, seed=341)
    inp = make_inputs(w, device="cuda")
    host = {k: (v if k in ("dt_bias", "A", "D") else _pinned(v)) for k, v in inp.items()}
    scratch = m.Workspace("cuda")
    y_e, f_e = m.ssd_fwd_host(**host, chunk_size=w.chunk, pieces=3, scratch=scratch)
    torch.cuda.synchronize()
    y_g = torch.zeros_like(y_e).pin_memory()
    f_g = torch.zeros_like(f_e).pin_memory()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        m.ssd_fwd_host(**host, chunk_size=w.chunk, pieces=3, scratch=scratch, y=y_g, final_states=f_g,
                       stream=stream)
    for _ in range(2):
        y_g.zero_()
        f_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        m.check(scratch)
        assert torch.equal(y_g, y_e) and torch.equal(f_g, f_e)


# ----------------------------------------------------------------------------- randomised shapes
def _random_cases(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        tc = i % 2 == 0  # alternate shapes the tensor-core kernel takes and shapes only the SIMT kernel takes
        H = int(rng.choice([2, 4, 6, 8]))
        G = int(rng.choice([g for g in (1, 2, 3, 4, 6, 8) if H % g == 0]))
        io = str(rng.choice(["bf16", "f16"])) if tc else str(rng.choice(["f32", "bf16", "f16"]))
        over = dict(batch=int(rng.integers(1, 4)), seqlen=int(rng.integers(1, 1300)), nheads=H, ngroups=G, io=io,
                    headdim=64 if tc else int(rng.choice([16, 32, 64])),
                    dstate=128 if tc else int(rng.choice([16, 32, 64, 128])),
                    chunk=int(rng.choice([128, 256])) if tc else int(rng.choice([32, 64, 128])),
                    state=str(rng.choice(["f32", "f16"])), init=str(rng.choice(["none", "normal"])), seed=5000 + i)
        cases.append(over)
    return cases


@pytest.mark.parametrize("over", _random_cases(), ids=[f"rand{i}" for i in range(24)])
def test_random_shapes_against_the_oracle(over):
    """Seeded random problems across both prefill kernels (and the decode step when a length of 1 comes up):
    batch, odd lengths, groups, head and state sizes, chunk sizes, dtypes, with and without initial states."""
    w = WORKLOADS["m130-bf16"].with_(**over)
    inp = make_inputs(w, device="cuda")
    y, fin = run_gpu(w, inp)
    yr, fr = oracle.ssd_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, f"random {over}")


def _random_varlen_cases(n=10, seed=2025):
    """Length mixes with empty, one-token, chunk-edge and long sequences, on both prefill kernels."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        tc = i % 2 == 0
        H = int(rng.choice([2, 4, 8]))
        G = int(rng.choice([g for g in (1, 2, 4) if H % g == 0]))
        chunk = int(rng.choice([128, 256])) if tc else int(rng.choice([32, 64]))
        pool = [0, 1, chunk - 1, chunk, chunk + 1] + [int(v) for v in rng.integers(2, 900, size=3)]
        lengths = [int(rng.choice(pool)) for _ in range(int(rng.integers(1, 7)))]
        over = dict(nheads=H, ngroups=G, chunk=chunk, io=str(rng.choice(["bf16", "f16"])),
                    state=str(rng.choice(["f32", "f16"])), init=str(rng.choice(["none", "normal"])),
                    headdim=64 if tc else int(rng.choice([32, 64])), dstate=128 if tc else int(rng.choice([32, 128])))
        cases.append(("tc" if tc else "simt", over, lengths, 7000 + i))
    return cases


@pytest.mark.parametrize("kernel,over,lengths,seed", _random_varlen_cases(), ids=[f"rvar{i}" for i in range(10)])
def test_random_varlen_against_the_oracle(kernel, over, lengths, seed):
    w = WORKLOADS["m130-bf16"].with_(**over)
    inp = make_varlen_inputs(w, lengths, device="cuda", seed=seed)
    ws = m.Workspace("cuda")
    y, fin = m.ssd_fwd_varlen(**inp, chunk_size=w.chunk, state_dtype=DTYPES[w.state], kernel=kernel, workspace=ws)
    m.check(ws)
    yr, fr = oracle.ssd_varlen_reference(**cpu(inp))
    assert_parity(w, y, fin, yr, fr, f"random varlen {kernel} {over} {lengths}", kernel=kernel)


def _random_conv_cases(n=8, seed=2026):
    """Conv widths 1 .. 8, both activations, with and without a cache, fused and unfused, prefill and one token."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        H = int(rng.choice([2, 4]))
        over = dict(batch=int(rng.integers(1, 4)), seqlen=int(rng.choice([1, int(rng.integers(2, 600))])), nheads=H,
                    ngroups=int(rng.choice([1, 2])), io=str(rng.choice(["bf16", "f16"])),
                    state=str(rng.choice(["f32", "f16"])), init=str(rng.choice(["none", "normal"])), seed=8000 + i)
        cases.append((over, int(rng.integers(1, 9)), str(rng.choice(["silu", "none"])), bool(rng.integers(0, 2)),
                      bool(rng.integers(0, 2))))
    return cases


@pytest.mark.parametrize("over,width,act,cache,fuse", _random_conv_cases(), ids=[f"rconv{i}" for i in range(8)])
def test_random_conv_against_the_oracle(over, width, act, cache, fuse):
    w = WORKLOADS["m130-bf16"].with_(**over)
    inp = make_conv_inputs(w, width, device="cuda", seed=w.seed, conv_state=cache)
    ws = m.Workspace("cuda")
    y, fin, cs, _ = m.ssd_fwd_conv(**inp, nheads=w.nheads, headdim=w.headdim, ngroups=w.ngroups, dstate=w.dstate,
                                   activation=act, chunk_size=w.chunk, state_dtype=DTYPES[w.state], workspace=ws,
                                   fuse=fuse)
    m.check(ws)
    yr, fr, csr = conv_reference(w, inp, width, act)
    assert_parity(w, y, fin, yr, fr, f"random conv {over} k={width} {act} cache={cache} fuse={fuse}")
    assert np.array_equal(cs.double().cpu().numpy(), csr)
