"""CPU oracle for the Mamba-2 SSD prefill forward.

TEST INFRASTRUCTURE ONLY: only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import this package. The CUDA library never
imports it, and it imports nothing from the CUDA library.

The arithmetic lives in ``ssd_oracle.c``: the fp64 token-by-token recurrence

    dt_t = softplus(dt_raw_t + dt_bias_h)
    h_t  = exp(dt_t * A_h) * h_{t-1} + dt_t * x_t (outer) B_t
    y_t  = C_t . h_t + D_h * x_t

run independently for every (batch, head) chain, with the head-to-group map
g = h // (H / G). This module only gathers each chain's slices, converts the
stored inputs exactly to float64, and calls the C code.

Page citations: the recurrence is the selective linear recurrence of "Mamba
hardware-aware algorithms" (section on the associative-scan foundations) with
the discretisation of "Mamba-2 compiler optimisation" section 1.1; the state
layout [B, H, P, N] is that page's decode-cache layout (section 2.2).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle's C source with the host compiler (gcc)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.oracle_ssd_chains.argtypes = [i64, i64, i64, i64, d, d, d, d, d, d, d, d, d, d, ctypes.c_int]
            lib.oracle_ssd_chains.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    """Exact conversion of a stored tensor (torch or numpy; f32/f16/bf16/f64) to float64 numpy."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        import torch

        return a.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def ssd_chains(x, dt_raw, dt_bias, A, B, C, D=None, init=None, nthreads=None):
    """Run stacked independent chains.

    x [n, L, P], dt_raw [n, L], dt_bias/A/D [n], B/C [n, L, N], init [n, P, N].
    Returns (y [n, L, P], final [n, P, N]) as float64 arrays.
    """
    x, dt_raw, dt_bias, A, B, C = (_f64(v) for v in (x, dt_raw, dt_bias, A, B, C))
    D, init = _f64(D), _f64(init)
    n, L, P = x.shape
    N = B.shape[-1]
    assert dt_raw.shape == (n, L) and B.shape == (n, L, N) and C.shape == (n, L, N)
    assert dt_bias.shape == (n,) and A.shape == (n,)
    assert D is None or D.shape == (n,)
    assert init is None or init.shape == (n, P, N)
    y = np.empty((n, L, P), dtype=np.float64)
    fin = np.empty((n, P, N), dtype=np.float64)
    rc = _load().oracle_ssd_chains(n, L, P, N, _ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C),
                                   _ptr(D), _ptr(init), _ptr(y), _ptr(fin), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_ssd_chains rejected its arguments")
    return y, fin


def ssd_reference(x, dt_raw, dt_bias, A, B, C, D=None, init_states=None, chains=None, nthreads=None):
    """Oracle SSD forward on library-layout inputs.

    x [b, L, H, P], dt_raw [b, L, H], dt_bias/A/D [H], B/C [b, L, G, N],
    init_states [b, H, P, N] (None = zeros). With ``chains`` None every (b, h)
    chain is run and (y [b, L, H, P], final [b, H, P, N]) is returned; with a
    list of (b, h) pairs only those run and (y [n, L, P], final [n, P, N]) is
    returned in the list's order.
    """
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if H % G:
        raise ValueError("nheads must be a multiple of ngroups")
    per = H // G
    all_chains = chains is None
    if all_chains:
        chains = [(bi, h) for bi in range(b) for h in range(H)]
    bs = np.array([c[0] for c in chains], dtype=np.int64)
    hs = np.array([c[1] for c in chains], dtype=np.int64)
    gs = hs // per
    if len(chains) == 0:
        return np.empty((0, L, P)), np.empty((0, P, N))

    # gather one chain at a time: keeps the exact conversion and the memory small
    xs = np.stack([_f64(x[int(bi), :, int(h), :]) for bi, h in zip(bs, hs)])
    dts = np.stack([_f64(dt_raw[int(bi), :, int(h)]) for bi, h in zip(bs, hs)])
    Bs = np.stack([_f64(B[int(bi), :, int(g), :]) for bi, g in zip(bs, gs)])
    Cs = np.stack([_f64(C[int(bi), :, int(g), :]) for bi, g in zip(bs, gs)])
    bias = _f64(dt_bias)[hs]
    Ah = _f64(A)[hs]
    Dh = None if D is None else _f64(D)[hs]
    init = None if init_states is None else np.stack([_f64(init_states[int(bi), int(h)]) for bi, h in zip(bs, hs)])
    y, fin = ssd_chains(xs, dts, bias, Ah, Bs, Cs, Dh, init, nthreads=nthreads)
    if not all_chains:
        return y, fin
    y_full = np.empty((b, L, H, P), dtype=np.float64)
    f_full = np.empty((b, H, P, N), dtype=np.float64)
    for k, (bi, h) in enumerate(chains):
        y_full[bi, :, h, :] = y[k]
        f_full[bi, h] = fin[k]
    return y_full, f_full


def ssd_varlen_reference(x, dt_raw, dt_bias, A, B, C, cu_seqlens, D=None, init_states=None, nthreads=None):
    """Oracle for a variable-length batch ("Mamba hardware-aware algorithms": sequences packed along one
    token axis, each its own recurrence). x [1, T, H, P], dt_raw [1, T, H], B/C [1, T, G, N], cu_seqlens
    [nseq + 1] token offsets, init_states [nseq, H, P, N] (None = zeros). Sequence s (tokens cu[s] .. cu[s+1])
    runs the plain recurrence from init_states[s]; a sequence of length 0 keeps its initial state.
    Returns (y [1, T, H, P], final [nseq, H, P, N]) as float64 arrays.
    """
    cu = [int(v) for v in np.asarray(cu_seqlens).reshape(-1)]
    nseq = len(cu) - 1
    _, T, H, P = x.shape
    N = B.shape[3]
    y = np.zeros((1, T, H, P), dtype=np.float64)
    fin = np.zeros((nseq, H, P, N), dtype=np.float64)
    for s in range(nseq):
        a, b = cu[s], cu[s + 1]
        init = None if init_states is None else init_states[s:s + 1]
        if b == a:
            if init is not None:
                fin[s] = _f64(init)[0]
            continue
        ys, fs = ssd_reference(x[:, a:b], dt_raw[:, a:b], dt_bias, A, B[:, a:b], C[:, a:b], D, init, nthreads=nthreads)
        y[0, a:b] = ys[0]
        fin[s] = fs[0]
    return y, fin


def conv1d_reference(xbc, weight, bias=None, conv_state=None, activation="silu"):
    """Causal depthwise convolution over the token axis ("Accelerating Mamba2 with Kernel Fusion": the depthwise
    convolution that mixes each channel's most recent tokens; "Mamba-2 compiler optimisation" section 2.2: the
    conv cache of the last k - 1 inputs per channel, [batch, channels, k - 1]).

    xbc [b, L, D] raw inputs, weight [D, k], bias [D] (None = 0), conv_state [b, D, k - 1] (None = zeros: the
    tokens before the sequence), activation "silu" (v * sigmoid(v)) or "none". For every channel ch:
        out[t, ch] = act(bias[ch] + sum_j weight[ch, j] * in[t - (k - 1) + j, ch])
    with in[t' < 0] taken from conv_state. Returns (out [b, L, D], state_out [b, D, k - 1]: the last k - 1 inputs,
    the cache for continuing the sequence) as float64 arrays.
    """
    x = _f64(xbc)
    w = _f64(weight)
    b, L, D = x.shape
    k = w.shape[1]
    prev = np.zeros((b, k - 1, D)) if conv_state is None else np.transpose(_f64(conv_state), (0, 2, 1))
    full = np.concatenate([prev, x], axis=1)  # [b, k - 1 + L, D]
    out = np.zeros((b, L, D))
    for j in range(k):
        out += w[None, None, :, j] * full[:, j:j + L, :]
    if bias is not None:
        out += _f64(bias)[None, None, :]
    if activation == "silu":
        out = out / (1.0 + np.exp(-out))
    elif activation != "none":
        raise ValueError("activation must be 'silu' or 'none'")
    state_out = np.transpose(full[:, L:, :], (0, 2, 1)).copy()  # the last k - 1 inputs
    return out, state_out


def ssd_conv_reference(xbc, weight, conv_bias, dt_raw, dt_bias, A, nheads, headdim, ngroups, dstate, D=None,
                       init_states=None, conv_state=None, activation="silu", nthreads=None):
    """The SSD forward on the output of the causal depthwise convolution: xbc [b, L, H*P + 2*G*N] raw, convolved
    (conv1d_reference), then split along channels into x [b, L, H, P], B and C [b, L, G, N], then ssd_reference.
    Returns (y, final_states, conv_state_out)."""
    out, state_out = conv1d_reference(xbc, weight, conv_bias, conv_state, activation)
    b, L, _ = out.shape
    hp, gn = nheads * headdim, ngroups * dstate
    x = out[:, :, :hp].reshape(b, L, nheads, headdim)
    B = out[:, :, hp:hp + gn].reshape(b, L, ngroups, dstate)
    C = out[:, :, hp + gn:hp + 2 * gn].reshape(b, L, ngroups, dstate)
    y, fin = ssd_reference(x, dt_raw, dt_bias, A, B, C, D, init_states, nthreads=nthreads)
    return y, fin, state_out
