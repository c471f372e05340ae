"""Cases for the bounds-checked debug build (run as a script by test_gpu_parity.py with MAMBA_SSD_LIB pointing at
libmamba_ssd_checked.so): every entry point on edge-case shapes, each followed by a status check, then the planted
probe, which must be reported. Prints one line per case: "<name> <status>" (0 = no violation)."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import mamba_ssd_prefill_gb300 as m  # noqa: E402
from mamba_ssd_prefill_gb300.inputs import WORKLOADS, DTYPES, make_conv_inputs, make_inputs, make_varlen_inputs  # noqa: E402

assert m.LIB_PATH.endswith("libmamba_ssd_checked.so"), m.LIB_PATH


def status(ws):
    try:
        m.check(ws)
        return 0
    except m.SsdError as e:
        return e.status


def run(name, fn):
    ws = m.Workspace("cuda")
    fn(ws)
    torch.cuda.synchronize()
    print(name, status(ws), flush=True)


def prefill(over, kernel="auto"):
    w = WORKLOADS["m130-bf16"].with_(**over)
    inp = make_inputs(w, device="cuda")
    return lambda ws: m.ssd_fwd(**inp, chunk_size=w.chunk, state_dtype=DTYPES[w.state], kernel=kernel, workspace=ws)


run("tc-ragged-2groups", prefill(dict(batch=2, seqlen=300, nheads=4, ngroups=2)))
run("tc-f16-states", prefill(dict(batch=1, seqlen=257, nheads=2, io="f16", state="f16")))
run("tc-chunk256-no-init", prefill(dict(batch=2, seqlen=700, nheads=4, chunk=256, init="none")))
run("simt-fp32", prefill(dict(batch=2, seqlen=333, nheads=3, io="f32", chunk=64), kernel="simt"))
run("simt-bf16", prefill(dict(batch=1, seqlen=200, nheads=2), kernel="simt"))
run("step-staged", prefill(dict(batch=7, seqlen=1, nheads=8)))
run("step-registers", prefill(dict(batch=3, seqlen=1, nheads=2, headdim=24, dstate=100)))
run("step-no-init", prefill(dict(batch=4, seqlen=1, nheads=4, init="none", state="f16")))

w = WORKLOADS["m130-bf16"].with_(nheads=4)
vl = make_varlen_inputs(w, [300, 0, 1, 129, 512], device="cuda", seed=3)
run("varlen-with-empty", lambda ws: m.ssd_fwd_varlen(**vl, chunk_size=128, workspace=ws))
vs = make_varlen_inputs(w.with_(io="f32"), [70, 0, 33], device="cuda", seed=4)
run("varlen-simt", lambda ws: m.ssd_fwd_varlen(**vs, chunk_size=64, kernel="simt", workspace=ws))

wc = WORKLOADS["m130-bf16"].with_(batch=2, seqlen=300, nheads=4)
ci = make_conv_inputs(wc, 4, device="cuda", seed=5)
kw = dict(nheads=wc.nheads, headdim=wc.headdim, ngroups=wc.ngroups, dstate=wc.dstate, chunk_size=wc.chunk)
run("conv-tiled", lambda ws: m.ssd_fwd_conv(**ci, **kw, workspace=ws))
run("conv-fused", lambda ws: m.ssd_fwd_conv(**ci, **kw, fuse=True, workspace=ws))
c3 = make_conv_inputs(wc.with_(batch=3, seqlen=130), 3, device="cuda", seed=6, conv_state=False)
run("conv-width3-no-cache", lambda ws: m.ssd_fwd_conv(**c3, **kw, workspace=ws))

wh = WORKLOADS["m130-bf16"].with_(batch=3, seqlen=650, nheads=4)
hi = make_inputs(wh, device="cuda")
host = {k: (v if k in ("dt_bias", "A", "D") else (None if v is None else v.cpu().pin_memory())) for k, v in hi.items()}
run("host-streaming", lambda ws: m.ssd_fwd_host(**host, chunk_size=wh.chunk, pieces=3, scratch=ws))

# the planted probe: the tensor-core kernel's dt_raw indices one extent too far must be caught and reported
wp = WORKLOADS["m130-bf16"].with_(batch=1, seqlen=256, nheads=2)
pi = make_inputs(wp, device="cuda")
ws = m.Workspace("cuda")
m.ssd_fwd(**pi, chunk_size=wp.chunk, workspace=ws)
m.check(ws)
m.debug_set(ws, skip_publish=-2)
m.ssd_fwd(**pi, chunk_size=wp.chunk, workspace=ws)
torch.cuda.synchronize()
print("probe", status(ws), flush=True)
m.debug_set(ws, skip_publish=-1)
m.ssd_fwd(**pi, chunk_size=wp.chunk, workspace=ws)
torch.cuda.synchronize()
print("after-probe", status(ws), flush=True)
