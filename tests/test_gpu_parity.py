"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element."""
import numpy as np
import pytest
import torch

import mamba_ssd_prefill_gb300 as m
import oracle
from mamba_ssd_prefill_gb300.inputs import DTYPES, WORKLOADS, make_inputs
from parity import gate_final, gate_y

pytestmark = pytest.mark.gpu


def cpu(d):
    return {k: (v.cpu() if v is not None else None) for k, v in d.items()}


def run_gpu(w, inp, kernel="auto", ws=None, **kw):
    ws = ws or m.Workspace("cuda")
    y, fin = m.ssd_fwd(**inp, chunk_size=w.chunk, state_dtype=DTYPES[w.state], kernel=kernel, workspace=ws, **kw)
    m.check(ws)
    return y, fin


def assert_parity(w, y, fin, yr, fr, label=""):
    ok, s = gate_y(y.double().cpu().numpy(), yr, w.io)
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
    assert_parity(w, y, fin, yr, fr, f"simt {name} {over}")


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
