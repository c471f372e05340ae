"""GB300-native Mamba-2 SSD chunked-scan prefill forward.

A thin ctypes binding over the C ABI in ``include/ssd.h`` (``libmamba_ssd.so``,
built in-tree by ``_build.py``). This module only marshals arguments: it
checks tensor shapes and dtypes, allocates outputs and the workspace with
PyTorch (device memory and streams are PyTorch's job here), and passes raw
pointers. Every step of the computation runs in the library's CUDA kernels;
there is no CPU path. If the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["ssd_fwd", "ssd_fwd_host", "ssd_fwd_varlen", "ssd_fwd_conv", "workspace_size", "make_problem", "check", "debug_set", "debug_knobs", "kernel_for", "plan_info", "SsdError",
           "Workspace", "lib", "LIB_PATH", "STATUS"]

# MAMBA_SSD_LIB selects another build of the library (the bounds-checked debug build, libmamba_ssd_checked.so)
LIB_PATH = os.environ.get("MAMBA_SSD_LIB") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmamba_ssd.so")

_DT = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
_KERNEL = {"auto": 0, "simt": 1, "tc": 2, "step": 3}
STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED", 3: "SSD_ERR_WORKSPACE",
          4: "SSD_ERR_CUDA", 5: "SSD_ERR_TIMEOUT", 6: "SSD_ERR_DEVICE"}


class SsdProblem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("chunk_size", ctypes.c_int64), ("io_dtype", ctypes.c_int32), ("state_dtype", ctypes.c_int32),
                ("kernel", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class SsdPlan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("launches", ctypes.c_int32), ("segments", ctypes.c_int64),
                ("segment_chunks", ctypes.c_int64), ("workspace_bytes", ctypes.c_size_t),
                ("head_flags", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class SsdError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = STATUS.get(status, str(status))
        text = _lib.ssd_status_string(status).decode() if _lib is not None else name
        super().__init__(f"{what}: {name} ({text})" if what else f"{name} ({text})")


_lib = None
_lock = threading.Lock()


def lib():
    """Load libmamba_ssd.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                                   f"g.build()'` (nvcc, sm_103a). There is no CPU fallback.")
            L = ctypes.CDLL(LIB_PATH)
            vp, sz, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64
            pp = ctypes.POINTER(SsdProblem)
            L.ssd_fwd_workspace_size.argtypes = [pp, ctypes.POINTER(sz)]
            L.ssd_fwd_workspace_size.restype = ctypes.c_int
            L.ssd_fwd.argtypes = [pp] + [vp] * 10 + [vp, sz, vp]
            L.ssd_fwd.restype = ctypes.c_int
            L.ssd_fwd_varlen_workspace_size.argtypes = [pp, i64, ctypes.POINTER(sz)]
            L.ssd_fwd_varlen_workspace_size.restype = ctypes.c_int
            L.ssd_fwd_varlen.argtypes = [pp, vp, i64] + [vp] * 10 + [vp, sz, vp]
            L.ssd_fwd_varlen.restype = ctypes.c_int
            L.ssd_fwd_conv.argtypes = [pp, ctypes.c_int32, ctypes.c_int32] + [vp] * 14 + [sz, vp]
            L.ssd_fwd_conv.restype = ctypes.c_int
            L.ssd_fwd_host_scratch_size.restype = ctypes.c_int
            L.ssd_fwd_host_scratch_size.argtypes = [pp, ctypes.c_int32, ctypes.POINTER(sz)]
            L.ssd_fwd_host.restype = ctypes.c_int
            L.ssd_fwd_host.argtypes = [pp, ctypes.c_int32] + [vp] * 10 + [vp, sz, vp]
            L.ssd_fwd_check.argtypes = [vp, vp]
            L.ssd_fwd_check.restype = ctypes.c_int
            L.ssd_debug_set.argtypes = [vp, ctypes.c_uint64, i64, vp]
            L.ssd_debug_set.restype = ctypes.c_int
            L.ssd_debug_knobs.argtypes = [ctypes.c_int32] * 6
            L.ssd_debug_knobs.restype = ctypes.c_int
            L.ssd_fwd_kernel_for.argtypes = [pp]
            L.ssd_fwd_kernel_for.restype = ctypes.c_int
            L.ssd_fwd_plan.argtypes = [pp, ctypes.POINTER(SsdPlan)]
            L.ssd_fwd_plan.restype = ctypes.c_int
            L.ssd_status_string.argtypes = [ctypes.c_int]
            L.ssd_status_string.restype = ctypes.c_char_p
            L.ssd_version.argtypes = []
            L.ssd_version.restype = ctypes.c_int
            _lib = L
    return _lib


def make_problem(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, io_dtype=torch.bfloat16,
                 state_dtype=torch.float32, kernel="auto") -> SsdProblem:
    return SsdProblem(int(batch), int(seqlen), int(nheads), int(headdim), int(dstate), int(ngroups), int(chunk_size),
                      _DT[io_dtype], _DT[state_dtype], _KERNEL[kernel], 0)


def workspace_size(prob: SsdProblem) -> int:
    n = ctypes.c_size_t(0)
    st = lib().ssd_fwd_workspace_size(ctypes.byref(prob), ctypes.byref(n))
    if st:
        raise SsdError(st, "ssd_fwd_workspace_size")
    return int(n.value)


def plan_info(prob: SsdProblem) -> dict:
    """What ssd_fwd plans for a regular batch: kernel, launches per call, segments, chunks per segment, workspace,
    and whether the tensor-core kernel passes states behind one release flag per head."""
    pl = SsdPlan()
    st = lib().ssd_fwd_plan(ctypes.byref(prob), ctypes.byref(pl))
    if st:
        raise SsdError(st, "ssd_fwd_plan")
    return {"kernel": {1: "simt", 2: "tc", 3: "step"}[pl.kernel], "launches": pl.launches, "segments": pl.segments,
            "segment_chunks": pl.segment_chunks, "workspace_bytes": pl.workspace_bytes,
            "head_flags": bool(pl.head_flags)}


def kernel_for(prob: SsdProblem) -> str:
    k = lib().ssd_fwd_kernel_for(ctypes.byref(prob))
    if k < 0:
        raise SsdError(-k, "ssd_fwd_kernel_for")
    return {1: "simt", 2: "tc", 3: "step"}[k]


class Workspace:
    """A zero-initialised device workspace, grown on demand and reused across calls on one stream."""

    # the state-passing tags carry the launch count modulo 2^22: the buffer is zero-filled again well before that
    REZERO_EVERY = 1 << 21

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = None
        self.calls = 0

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            # the library asks for a zero-filled workspace on first use only
            self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)
            self.calls = 0
        self.calls += 1
        if self.calls % self.REZERO_EVERY == 0:
            self.buf.zero_()  # on the current stream, ordered before the call that uses it
        return self.buf


_default_ws: dict = {}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def ssd_fwd(x, dt_raw, dt_bias, A, B, C, D=None, init_states=None, chunk_size=128, state_dtype=None, *, y=None,
            final_states=None, return_final_states=True, workspace=None, kernel="auto", stream=None):
    """Fused Mamba-2 SSD prefill forward on the GPU.

    x [b, L, H, P], dt_raw [b, L, H], B/C [b, L, G, N] in one I/O dtype (fp32,
    bf16 or fp16); dt_bias, A, D [H] fp32; init_states [b, H, P, N] in the
    state dtype (fp32 or fp16). Returns (y [b, L, H, P], final_states or None).
    """
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("ssd_fwd runs on CUDA tensors only (there is no CPU path)")
    io = x.dtype
    if state_dtype is None:
        state_dtype = init_states.dtype if init_states is not None else torch.float32
    for name, t, shape, dt in (("dt_raw", dt_raw, (b, L, H), io), ("B", B, (b, L, G, N), io), ("C", C, (b, L, G, N), io),
                               ("dt_bias", dt_bias, (H,), torch.float32), ("A", A, (H,), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dt or t.device != dev or not t.is_contiguous():
            raise ValueError(f"{name}: expected contiguous {dt} {shape} on {dev}, got {t.dtype} {tuple(t.shape)}")
    if D is not None and (tuple(D.shape) != (H,) or D.dtype != torch.float32 or not D.is_contiguous()):
        raise ValueError("D: expected contiguous fp32 [H]")
    if init_states is not None and (tuple(init_states.shape) != (b, H, P, N) or init_states.dtype != state_dtype
                                    or not init_states.is_contiguous()):
        raise ValueError("init_states: expected contiguous [b, H, P, N] in the state dtype")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    prob = make_problem(b, L, H, P, N, G, chunk_size, io, state_dtype, kernel)
    nbytes = workspace_size(prob)
    if y is None:
        y = torch.empty_like(x)
    if final_states is None and return_final_states:
        final_states = torch.empty(b, H, P, N, dtype=state_dtype, device=dev)
    if workspace is None:
        key = (dev.index, torch.cuda.current_stream(dev).cuda_stream if stream is None else stream.cuda_stream)
        workspace = _default_ws.setdefault(key, Workspace(dev))
    ws = workspace.get(nbytes) if isinstance(workspace, Workspace) else workspace
    st = lib().ssd_fwd(ctypes.byref(prob), _ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                       _ptr(init_states), _ptr(y), _ptr(final_states), _ptr(ws), ws.numel() * ws.element_size(),
                       _stream_ptr(stream, dev))
    if st:
        raise SsdError(st, "ssd_fwd")
    return y, final_states


def ssd_fwd_host(x, dt_raw, dt_bias, A, B, C, D=None, init_states=None, chunk_size=128, state_dtype=None, *,
                 pieces=0, y=None, final_states=None, return_final_states=True, scratch=None, kernel="auto",
                 stream=None):
    """The forward pass on host-resident tensors, streamed through the GPU in token pieces of the whole batch (the
    copies of one piece overlap the computation of another; pieces=0 lets the library choose). x, dt_raw, B, C, init_states and the outputs are CPU tensors (page-locked
    for the overlap: the outputs are allocated page-locked when not given); dt_bias, A, D are CUDA tensors and
    choose the device. `scratch` is a Workspace (its buffer starts with the workspace that check() reads). The call
    is asynchronous on `stream`: synchronise it before reading y and the final states."""
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev = dt_bias.device
    if dev.type != "cuda":
        raise ValueError("ssd_fwd_host: dt_bias, A, D are CUDA tensors (the computation runs on that GPU)")
    io = x.dtype
    if state_dtype is None:
        state_dtype = init_states.dtype if init_states is not None else torch.float32
    for name, t, shape, dt in (("x", x, (b, L, H, P), io), ("dt_raw", dt_raw, (b, L, H), io),
                               ("B", B, (b, L, G, N), io), ("C", C, (b, L, G, N), io)):
        if tuple(t.shape) != shape or t.dtype != dt or t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous CPU {dt} {shape}, got {t.dtype} {tuple(t.shape)} "
                             f"on {t.device}")
    for name, t in (("dt_bias", dt_bias), ("A", A), ("D", D)):
        if t is not None and (tuple(t.shape) != (H,) or t.dtype != torch.float32 or t.device != dev
                              or not t.is_contiguous()):
            raise ValueError(f"{name}: expected a contiguous fp32 [H] tensor on {dev}")
    if init_states is not None and (tuple(init_states.shape) != (b, H, P, N) or init_states.dtype != state_dtype
                                    or init_states.device.type != "cpu" or not init_states.is_contiguous()):
        raise ValueError("init_states: expected a contiguous CPU [b, H, P, N] tensor in the state dtype")
    prob = make_problem(b, L, H, P, N, G, chunk_size, io, state_dtype, kernel)
    n = ctypes.c_size_t(0)
    st = lib().ssd_fwd_host_scratch_size(ctypes.byref(prob), int(pieces), ctypes.byref(n))
    if st:
        raise SsdError(st, "ssd_fwd_host_scratch_size")
    if y is None:
        y = torch.empty(x.shape, dtype=io, pin_memory=True)
    if final_states is None and return_final_states:
        final_states = torch.empty(b, H, P, N, dtype=state_dtype, pin_memory=True)
    for name, t in (("y", y), ("final_states", final_states)):
        if t is not None and (t.device.type != "cpu" or not t.is_contiguous()):
            raise ValueError(f"{name}: expected a contiguous CPU tensor")
    if scratch is None:
        key = ("host", dev.index, torch.cuda.current_stream(dev).cuda_stream if stream is None else stream.cuda_stream)
        scratch = _default_ws.setdefault(key, Workspace(dev))
    buf = scratch.get(n.value) if isinstance(scratch, Workspace) else scratch
    with torch.cuda.device(dev):
        st = lib().ssd_fwd_host(ctypes.byref(prob), int(pieces), _ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(A),
                                _ptr(B), _ptr(C), _ptr(D), _ptr(init_states), _ptr(y), _ptr(final_states), _ptr(buf),
                                buf.numel() * buf.element_size(), _stream_ptr(stream, dev))
    if st:
        raise SsdError(st, "ssd_fwd_host")
    return y, final_states


def ssd_fwd_varlen(x, dt_raw, dt_bias, A, B, C, cu_seqlens, D=None, init_states=None, chunk_size=128,
                   state_dtype=None, *, y=None, final_states=None, return_final_states=True, workspace=None,
                   kernel="auto", stream=None):
    """Variable-length batch: nseq sequences packed along the token axis of x [1, T, H, P] (dt_raw [1, T, H],
    B/C [1, T, G, N]); cu_seqlens is an int32 CUDA tensor [nseq + 1] of token offsets. init_states and the
    returned final states are [nseq, H, P, N]. Offsets are checked on the device (see check())."""
    if x.dim() != 4 or x.shape[0] != 1:
        raise ValueError("x: expected [1, T, H, P] (sequences packed along T)")
    _, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("ssd_fwd_varlen runs on CUDA tensors only (there is no CPU path)")
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.device != dev or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1 \
            or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens: expected a contiguous int32 [nseq + 1] tensor on the device of x")
    nseq = cu_seqlens.numel() - 1
    io = x.dtype
    if state_dtype is None:
        state_dtype = init_states.dtype if init_states is not None else torch.float32
    for name, t, shape, dt in (("dt_raw", dt_raw, (1, T, H), io), ("B", B, (1, T, G, N), io), ("C", C, (1, T, G, N), io),
                               ("dt_bias", dt_bias, (H,), torch.float32), ("A", A, (H,), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dt or t.device != dev or not t.is_contiguous():
            raise ValueError(f"{name}: expected contiguous {dt} {shape} on {dev}, got {t.dtype} {tuple(t.shape)}")
    if D is not None and (tuple(D.shape) != (H,) or D.dtype != torch.float32 or not D.is_contiguous()):
        raise ValueError("D: expected contiguous fp32 [H]")
    if init_states is not None and (tuple(init_states.shape) != (nseq, H, P, N) or init_states.dtype != state_dtype
                                    or not init_states.is_contiguous()):
        raise ValueError("init_states: expected contiguous [nseq, H, P, N] in the state dtype")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    prob = make_problem(1, T, H, P, N, G, chunk_size, io, state_dtype, kernel)
    n = ctypes.c_size_t(0)
    st = lib().ssd_fwd_varlen_workspace_size(ctypes.byref(prob), nseq, ctypes.byref(n))
    if st:
        raise SsdError(st, "ssd_fwd_varlen_workspace_size")
    if y is None:
        y = torch.empty_like(x)
    if final_states is None and return_final_states:
        final_states = torch.empty(nseq, H, P, N, dtype=state_dtype, device=dev)
    if workspace is None:
        key = (dev.index, torch.cuda.current_stream(dev).cuda_stream if stream is None else stream.cuda_stream)
        workspace = _default_ws.setdefault(key, Workspace(dev))
    ws = workspace.get(int(n.value)) if isinstance(workspace, Workspace) else workspace
    st = lib().ssd_fwd_varlen(ctypes.byref(prob), _ptr(cu_seqlens), nseq, _ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(A),
                              _ptr(B), _ptr(C), _ptr(D), _ptr(init_states), _ptr(y), _ptr(final_states), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream_ptr(stream, dev))
    if st:
        raise SsdError(st, "ssd_fwd_varlen")
    return y, final_states


_ACT = {"none": 0, "silu": 1}


def ssd_fwd_conv(xbc, conv_weight, dt_raw, dt_bias, A, nheads, headdim, ngroups, dstate, conv_bias=None, D=None,
                 init_states=None, conv_state=None, activation="silu", chunk_size=128, state_dtype=None, *,
                 fuse=False, xbc_out=None, conv_state_out=None, return_conv_state=True, y=None, final_states=None,
                 return_final_states=True, workspace=None, kernel="auto", stream=None):
    """Causal depthwise convolution over the tokens, then the SSD on x | B | C column slices of its output.

    xbc [b, L, H*P + 2*G*N] raw (I/O dtype), conv_weight [D, k] fp32, conv_bias [D] fp32, conv_state
    [b, D, k-1] (None: a fresh sequence). By default the convolved rows are written to xbc_out first (the faster
    path on this kernel); with fuse (and no xbc_out) the tensor-core kernel convolves as it loads and no activation
    buffer exists (xbc_out returned None). Returns (y, final_states, conv_state_out, xbc_out)."""
    b, L, Dc = xbc.shape
    H, P, G, N = int(nheads), int(headdim), int(ngroups), int(dstate)
    dev = xbc.device
    if dev.type != "cuda":
        raise ValueError("ssd_fwd_conv runs on CUDA tensors only (there is no CPU path)")
    if Dc != H * P + 2 * G * N:
        raise ValueError("xbc: the channel count must be nheads*headdim + 2*ngroups*dstate")
    io = xbc.dtype
    k = conv_weight.shape[1]
    if state_dtype is None:
        state_dtype = init_states.dtype if init_states is not None else torch.float32
    for name, t, shape, dt in (("conv_weight", conv_weight, (Dc, k), torch.float32), ("dt_raw", dt_raw, (b, L, H), io),
                               ("dt_bias", dt_bias, (H,), torch.float32), ("A", A, (H,), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dt or t.device != dev or not t.is_contiguous():
            raise ValueError(f"{name}: expected contiguous {dt} {shape} on {dev}, got {t.dtype} {tuple(t.shape)}")
    for name, t, shape, dt in (("conv_bias", conv_bias, (Dc,), torch.float32), ("D", D, (H,), torch.float32),
                               ("conv_state", conv_state, (b, Dc, k - 1), io),
                               ("init_states", init_states, (b, H, P, N), state_dtype)):
        if t is not None and (tuple(t.shape) != shape or t.dtype != dt or t.device != dev or not t.is_contiguous()):
            raise ValueError(f"{name}: expected contiguous {dt} {shape} on {dev}")
    if not xbc.is_contiguous():
        raise ValueError("xbc must be contiguous")
    prob = make_problem(b, L, H, P, N, G, chunk_size, io, state_dtype, kernel)
    nbytes = workspace_size(prob)
    if xbc_out is None and not fuse:
        xbc_out = torch.empty_like(xbc)
    if conv_state_out is None and return_conv_state:
        conv_state_out = torch.empty(b, Dc, k - 1, dtype=io, device=dev)
    if y is None:
        y = torch.empty(b, L, H, P, dtype=io, device=dev)
    if final_states is None and return_final_states:
        final_states = torch.empty(b, H, P, N, dtype=state_dtype, device=dev)
    if workspace is None:
        key = (dev.index, torch.cuda.current_stream(dev).cuda_stream if stream is None else stream.cuda_stream)
        workspace = _default_ws.setdefault(key, Workspace(dev))
    ws = workspace.get(nbytes) if isinstance(workspace, Workspace) else workspace

    def call(out):
        return lib().ssd_fwd_conv(ctypes.byref(prob), int(k), _ACT[activation], _ptr(xbc), _ptr(conv_weight),
                                  _ptr(conv_bias), _ptr(conv_state), _ptr(conv_state_out), _ptr(out), _ptr(dt_raw),
                                  _ptr(dt_bias), _ptr(A), _ptr(D), _ptr(init_states), _ptr(y), _ptr(final_states),
                                  _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream, dev))

    st = call(xbc_out)
    if st == 2 and xbc_out is None:  # no fused instance for this problem: convolve into a buffer first
        xbc_out = torch.empty_like(xbc)
        st = call(xbc_out)
    if st:
        raise SsdError(st, "ssd_fwd_conv")
    return y, final_states, conv_state_out, xbc_out


def check(workspace, stream=None):
    """Synchronise and raise SsdError if a device-side wait failed in an earlier call."""
    ws = workspace.buf if isinstance(workspace, Workspace) else workspace
    if ws is None:
        return
    st = lib().ssd_fwd_check(_ptr(ws), _stream_ptr(stream, ws.device))
    if st:
        raise SsdError(st, "ssd_fwd_check")


def debug_set(workspace, timeout_ns=0, skip_publish=-1, stream=None):
    """Test hook: set the device wait limit and the chunk whose publish is skipped."""
    ws = workspace.buf if isinstance(workspace, Workspace) else workspace
    st = lib().ssd_debug_set(_ptr(ws), int(timeout_ns), int(skip_publish), _stream_ptr(stream, ws.device))
    if st:
        raise SsdError(st, "ssd_debug_set")


def debug_knobs(tc_heads_per_unit=-1, tc_late_ticket=-1, simt_two_pass=-1, conv_tma=-1, tc_segment_chunks=-1,
                tc_head_flags=-1):
    """Test hook: force launch-configuration choices of later calls (-1 everywhere restores the library's own).
    tc_segment_chunks changes the workspace size: allocate the workspace after setting it."""
    st = lib().ssd_debug_knobs(int(tc_heads_per_unit), int(tc_late_ticket), int(simt_two_pass), int(conv_tma),
                               int(tc_segment_chunks), int(tc_head_flags))
    if st:
        raise SsdError(st, "ssd_debug_knobs")
