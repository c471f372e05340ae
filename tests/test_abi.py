"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/ssd.h declares, and rejects bad problems before any
CUDA call."""
import ctypes
import os
import re

import pytest
import torch

import mamba_ssd_prefill_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"SSD_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(m.LIB_PATH):
        from mamba_ssd_prefill_gb300 import _build

        _build.build()
    return m.lib()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "ssd_fwd" in names and "ssd_fwd_workspace_size" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_version_and_status_strings(lib):
    assert lib.ssd_version() >= 10000
    for code in range(7):
        assert lib.ssd_status_string(code)


def prob(**kw):
    d = dict(batch=1, seqlen=1024, nheads=8, headdim=64, dstate=128, ngroups=1, chunk_size=128,
             io_dtype=torch.bfloat16, state_dtype=torch.float32, kernel="auto")
    d.update(kw)
    return m.make_problem(**d)


@pytest.mark.parametrize("bad", [dict(nheads=6, ngroups=4), dict(nheads=0), dict(chunk_size=0), dict(seqlen=-1),
                                 dict(headdim=0), dict(dstate=0)])
def test_rejects_bad_problem(lib, bad):
    with pytest.raises(m.SsdError) as e:
        m.workspace_size(prob(**bad))
    assert e.value.status == 1


def test_rejects_bad_enums(lib):
    p = prob()
    p.io_dtype = 7
    n = ctypes.c_size_t()
    assert lib.ssd_fwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 1
    p = prob()
    p.state_dtype = 1  # bf16 states are not offered
    assert lib.ssd_fwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 1
    p = prob()
    p.reserved = 3
    assert lib.ssd_fwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 1


def test_workspace_size_scales_with_chains(lib):
    a = m.workspace_size(prob(batch=1))
    b = m.workspace_size(prob(batch=4))
    assert b > a > 256
    assert a % 256 == 0


def test_kernel_selection(lib):
    assert m.kernel_for(prob(io_dtype=torch.float32, dstate=64)) == "simt"
    assert m.kernel_for(prob()) == "tc"
    assert m.kernel_for(prob(chunk_size=256)) == "tc"  # served in 128-token chunks
    assert m.kernel_for(prob(chunk_size=192)) == "simt"
    assert m.kernel_for(prob(chunk_size=64)) == "simt"
    assert m.kernel_for(prob(seqlen=1)) == "step"  # decode: one token advances the cached state
    assert m.kernel_for(prob(seqlen=1, kernel="tc")) == "tc"
    assert m.kernel_for(prob(seqlen=0, kernel="step")) == "step"
    with pytest.raises(m.SsdError) as e:
        m.kernel_for(prob(seqlen=2, kernel="step"))
    assert e.value.status == 2
    assert m.workspace_size(prob(seqlen=1)) == 256  # the header only
    assert m.kernel_for(prob(kernel="simt")) == "simt"
    # shapes the SIMT kernel cannot hold in shared memory are rejected
    with pytest.raises(m.SsdError) as e:
        m.kernel_for(prob(headdim=1024, dstate=1024, kernel="simt"))
    assert e.value.status == 2


def test_null_pointers_rejected_before_any_cuda_call(lib):
    p = prob(seqlen=64)
    vp = ctypes.c_void_p
    st = lib.ssd_fwd(ctypes.byref(p), None, None, None, None, None, None, None, None, None, None, None, 0, None)
    assert st == 1
    # misaligned x
    st = lib.ssd_fwd(ctypes.byref(p), vp(8), vp(256), vp(256), vp(256), vp(256), vp(256), None, None, vp(256), None,
                     vp(256), 1 << 30, None)
    assert st == 1


def test_workspace_rejected_when_small(lib):
    p = prob(seqlen=64)
    vp = ctypes.c_void_p
    a = vp(1 << 20)
    st = lib.ssd_fwd(ctypes.byref(p), a, a, a, a, a, a, None, None, a, None, a, 16, None)
    assert st == 3
    st = lib.ssd_fwd(ctypes.byref(p), a, a, a, a, a, a, None, None, a, None, vp((1 << 20) + 16), 1 << 30, None)
    assert st == 3


def test_python_binding_refuses_cpu_tensors(lib):
    x = torch.zeros(1, 4, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        m.ssd_fwd(x, torch.zeros(1, 4, 2, dtype=torch.bfloat16), torch.zeros(2), torch.zeros(2),
                  torch.zeros(1, 4, 1, 128, dtype=torch.bfloat16), torch.zeros(1, 4, 1, 128, dtype=torch.bfloat16))


def test_new_entry_points_reject_bad_arguments_before_any_cuda_call(lib):
    """The binding's argument lists match the C signatures (a wrong count raises TypeError here), and argument
    errors return before anything is launched."""
    p = prob(seqlen=64)
    assert lib.ssd_fwd_conv(ctypes.byref(p), 0, 1, *([None] * 14), 0, None) == 1       # conv width 0
    assert lib.ssd_fwd_conv(ctypes.byref(p), 4, 7, *([None] * 14), 0, None) == 1       # unknown activation
    assert lib.ssd_fwd_varlen(ctypes.byref(prob(batch=1)), None, -1, *([None] * 10), None, 0, None) == 1
    assert lib.ssd_fwd_varlen(ctypes.byref(prob(batch=2)), None, 3, *([None] * 10), None, 0, None) == 1  # batch != 1
    n = ctypes.c_size_t()
    assert lib.ssd_fwd_varlen_workspace_size(ctypes.byref(prob(batch=1)), 4, ctypes.byref(n)) == 0 and n.value > 256


def test_host_streaming_plan_and_argument_checks(lib):
    """ssd_fwd_host: the scratch holds the workspace of a piece, two slots of a piece's inputs and outputs and
    the states carried from piece to piece, so more pieces need less of it; argument errors return before any
    CUDA call."""
    n1, n4, n8 = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    p = prob(batch=3, seqlen=1024)
    assert lib.ssd_fwd_host_scratch_size(ctypes.byref(p), 1, ctypes.byref(n1)) == 0
    assert lib.ssd_fwd_host_scratch_size(ctypes.byref(p), 4, ctypes.byref(n4)) == 0
    assert lib.ssd_fwd_host_scratch_size(ctypes.byref(p), 8, ctypes.byref(n8)) == 0
    assert n1.value > n4.value > n8.value > 0
    # 4 pieces of 256 tokens: the workspace of [3, 256], three slots (x, y, dt_raw, B, C), the [3, H, P, N] states
    ws = ctypes.c_size_t()
    assert lib.ssd_fwd_workspace_size(ctypes.byref(prob(batch=3, seqlen=256)), ctypes.byref(ws)) == 0
    tok = 3 * 256
    slot = 2 * tok * 8 * 64 * 2 + tok * 8 * 2 + 2 * tok * 1 * 128 * 2
    assert n4.value >= ws.value + 3 * slot + 3 * 8 * 64 * 128 * 4
    # no more pieces than chunks
    n9, n99 = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.ssd_fwd_host_scratch_size(ctypes.byref(prob(batch=1, seqlen=1000)), 8, ctypes.byref(n9)) == 0
    assert lib.ssd_fwd_host_scratch_size(ctypes.byref(prob(batch=1, seqlen=1000)), 99, ctypes.byref(n99)) == 0
    assert n9.value == n99.value
    # from 8 pieces on the end pieces are short: 32 chunks in 8 pieces are 1, 5, 5, 5, 5, 5, 5, 1 chunks, so a slot
    # holds 5 chunks (640 tokens), between the even cuts into 8 (4 chunks) and 4 (8 chunks) pieces
    t8, t6, t4, ws5 = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    long = prob(batch=1, seqlen=32 * 128)
    assert lib.ssd_fwd_host_scratch_size(ctypes.byref(long), 8, ctypes.byref(t8)) == 0
    assert lib.ssd_fwd_host_scratch_size(ctypes.byref(long), 6, ctypes.byref(t6)) == 0
    assert lib.ssd_fwd_host_scratch_size(ctypes.byref(long), 4, ctypes.byref(t4)) == 0
    assert lib.ssd_fwd_workspace_size(ctypes.byref(prob(batch=1, seqlen=640)), ctypes.byref(ws5)) == 0
    tok = 640
    slot5 = 2 * tok * 8 * 64 * 2 + tok * 8 * 2 + 2 * tok * 1 * 128 * 2
    assert t8.value >= ws5.value + 3 * slot5 + 8 * 64 * 128 * 4
    assert t6.value > t8.value and t4.value > t8.value  # 6 pieces: an even cut of 6 chunks each
    assert lib.ssd_fwd_host_scratch_size(ctypes.byref(p), -1, ctypes.byref(n1)) == 1      # negative piece count
    assert lib.ssd_fwd_host(ctypes.byref(p), -1, *([None] * 10), None, 0, None) == 1
    assert lib.ssd_fwd_host(ctypes.byref(p), 0, *([None] * 10), None, 0, None) == 3       # no scratch
    bad = prob(batch=2, seqlen=64)
    bad.nheads = 3                                                                        # not a multiple of G
    bad.ngroups = 2
    assert lib.ssd_fwd_host_scratch_size(ctypes.byref(bad), 0, ctypes.byref(n1)) == 1


def test_bounds_checked_build_compiles_and_exports_every_symbol():
    """The bounds-checked debug library (SSD_BOUNDS_CHECK) builds from the same sources and exports the same C ABI;
    the GPU test runs it."""
    from mamba_ssd_prefill_gb300 import _build

    path = _build.build(checked=True)
    L = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(L, name), name


def test_debug_knobs_validate_and_restore(lib):
    """The launch-configuration test hooks take -1 (the library's choice) or a valid value, and reject the rest
    without changing anything."""
    assert lib.ssd_debug_knobs(-1, -1, -1, -1, -1, -1) == 0
    for bad in [(0, -1, -1, -1, -1, -1), (9, -1, -1, -1, -1, -1), (-1, 2, -1, -1, -1, -1), (-1, -1, -2, -1, -1, -1),
                (-1, -1, -1, 5, -1, -1), (-1, -1, -1, -1, -2, -1), (-1, -1, -1, -1, -1, 2), (-1, -1, -1, -1, -1, -2)]:
        assert lib.ssd_debug_knobs(*bad) == 1, bad
    assert lib.ssd_debug_knobs(8, 1, 0, 0, 4, 1) == 0
    m.debug_knobs()  # restore
    with pytest.raises(m.SsdError):
        m.debug_knobs(tc_heads_per_unit=0)


def test_library_sources_read_no_environment():
    """Launch choices come from the problem and the explicit test hooks only: no kernel or host file of the
    library reads an environment variable."""
    csrc = os.path.join(ROOT, "mamba_ssd_prefill_gb300", "csrc")
    for fn in os.listdir(csrc):
        src = open(os.path.join(csrc, fn)).read()
        assert "getenv" not in src, fn


def test_segment_knob_sizes_the_workspace(lib):
    """Two-level state passing (forced through the test hook) adds the segment entering states, the block
    aggregates and one state ring per segment to the workspace; a segment as long as the sequence changes nothing."""
    p = prob(batch=2, seqlen=4096, nheads=8, ngroups=2)  # 32 chunks per sequence
    base = m.workspace_size(p)
    try:
        m.debug_knobs(tc_segment_chunks=32)
        assert m.workspace_size(p) == base
        m.debug_knobs(tc_segment_chunks=8)  # 4 segments
        seg = m.workspace_size(p)
    finally:
        m.debug_knobs()
    state = 64 * 128 * 4
    entering = 2 * 3 * 8 * state           # sequences x (segments - 1) x heads
    assert seg >= base + entering + 2 * 3 * 8 * state  # at least one aggregate block per segment boundary
    assert m.workspace_size(p) == base


def test_segment_length_without_a_block_length_keeps_one_chain(lib):
    """A segment length with no block length in [8, 32] dividing it (683, a prime) cannot be cut into block units
    of whole chunks: the plan keeps one chain per sequence instead of a configuration the block kernel rejects."""
    p = prob(batch=1, seqlen=262144, nheads=80, ngroups=8)  # 2048 chunks
    try:
        m.debug_knobs(tc_segment_chunks=683)
        info = m.plan_info(p)
        assert info["segments"] == 1 and info["launches"] == 1 and info["segment_chunks"] == 2048
        m.debug_knobs(tc_segment_chunks=688)  # a multiple of 8: 3 segments
        info = m.plan_info(p)
        assert info["segments"] == 3 and info["segment_chunks"] == 688 and info["launches"] == 3
    finally:
        m.debug_knobs()


def test_host_pieces_sized_by_bytes(lib):
    """ssd_fwd_host's own piece count: about 256 MiB of copies a piece, from 8 to 32 pieces. The scratch of the
    library's choice equals that of the piece count it picks: 8 for a 2 GB batch, 25 for the 256K-token layer
    (6.5 GB of copies), 32 at most."""
    def scratch(p, pieces):
        n = ctypes.c_size_t(0)
        assert lib.ssd_fwd_host_scratch_size(ctypes.byref(p), pieces, ctypes.byref(n)) == 0
        return n.value
    small = prob(batch=8, seqlen=8192, nheads=80)  # 1.4 GB of copies
    assert scratch(small, 0) == scratch(small, 8) != scratch(small, 16)
    long = prob(batch=1, seqlen=262144, nheads=80, ngroups=8)  # 6.5 GB of copies
    assert scratch(long, 0) == scratch(long, 25) != scratch(long, 24)
    huge = prob(batch=8, seqlen=262144, nheads=80, ngroups=8)  # 52 GB of copies
    assert scratch(huge, 0) == scratch(huge, 32)


def test_plan_query_reports_kernel_launches_and_segments(lib):
    """ssd_fwd_plan: the kernel, the launches of one call (three with two-level state passing: block aggregates,
    their combination, the fused kernel) and the segments, consistent with ssd_fwd_workspace_size."""
    p = prob(batch=2, seqlen=4096, nheads=8, ngroups=2)  # 32 chunks
    info = m.plan_info(p)
    assert info["kernel"] == "tc" and info["segments"] == 1 and info["launches"] == 1
    assert info["segment_chunks"] == 32 and info["workspace_bytes"] == m.workspace_size(p)
    try:  # the per-head flag choice is reported as planned (forced both ways through the test hook)
        for forced in (0, 1):
            m.debug_knobs(tc_head_flags=forced)
            assert m.plan_info(p)["head_flags"] == bool(forced)
    finally:
        m.debug_knobs()
    assert not m.plan_info(prob(io_dtype=torch.float32, dstate=64))["head_flags"]  # SIMT kernel: no such flags
    try:
        m.debug_knobs(tc_segment_chunks=5)  # 32 chunks: 7 segments, the last of 2 chunks
        info = m.plan_info(p)
        assert info["segments"] == 7 and info["segment_chunks"] == 5 and info["launches"] == 3
        assert info["workspace_bytes"] == m.workspace_size(p)
    finally:
        m.debug_knobs()
    assert m.plan_info(prob(seqlen=1))["kernel"] == "step"
    assert m.plan_info(prob(seqlen=0, kernel="tc"))["launches"] == 0
    assert m.plan_info(prob(io_dtype=torch.float32, dstate=64))["kernel"] == "simt"
