"""Independent NumPy formulations of the SSD forward, used to pin the oracle.

None of these calls the oracle; each restates the method from a different
angle so that a mistake in the oracle's recurrence (a dropped term, a wrong
sign, a transposed outer product) shows up as a mismatch.

All functions work on ONE chain in float64:
  x [T, P], dt [T] (already discretised step sizes), A scalar, B, C [T, N],
  D scalar, h0 [P, N]. They return (y [T, P], final [P, N]).
"""
from __future__ import annotations

import numpy as np


def softplus(v):
    v = np.asarray(v, dtype=np.float64)
    return np.maximum(v, 0.0) + np.log1p(np.exp(-np.abs(v)))


def segsum(a):
    """Segment sums of a 1-D log-decay sequence, -inf above the diagonal.

    out[i, j] = a[j+1] + ... + a[i] for j <= i (0 on the diagonal), -inf for
    j > i: the stable log-space segment sum of "Mamba hardware-aware
    algorithms", section "Mamba-2 segsum stabilisation", taken as cumulative
    sum differences with a lower-triangular mask.
    """
    cs = np.cumsum(a)
    out = cs[:, None] - cs[None, :]
    T = a.shape[0]
    return np.where(np.tril(np.ones((T, T), dtype=bool)), out, -np.inf)


def quadratic(x, dt, A, B, C, D, h0):
    """Brute-force quadratic (attention-like) SSD with the materialised L o CB^T matrix.

    y = (exp(segsum(dt*A)) o (C B^T)) (dt o x) + exp(cumsum(dt*A)) o (C h0^T) + D x
    final = exp(cs_T) h0 + sum_s exp(cs_T - cs_s) dt_s x_s (outer) B_s
    ("Mamba hardware-aware algorithms", structured state space duality; the
    semiseparable matrix of the SSD framework.)
    """
    dA = dt * A
    Lmat = np.exp(segsum(dA))
    M = Lmat * (C @ B.T)
    cs = np.cumsum(dA)
    y = M @ (dt[:, None] * x) + np.exp(cs)[:, None] * (C @ h0.T) + D * x
    if len(dt):
        w = np.exp(cs[-1] - cs) * dt
        final = np.exp(cs[-1]) * h0 + (w[:, None] * x).T @ B
    else:
        final = h0.copy()
    return y, final


def chunked(x, dt, A, B, C, D, h0, Q):
    """The five SSD steps, chunk by chunk, exactly as the fused-kernel page lists them.

    chunk cumsum -> BMM (C B^T per chunk) -> chunk state (each chunk's end
    state from zero) -> state passing (global state at each chunk end) ->
    chunk scan (y from the chunk's x and the previous global state).
    ("Accelerating Mamba2 with Kernel Fusion", the SSD core operations.)
    """
    T, P = x.shape
    y = np.zeros_like(x)
    S = h0.copy()
    for c0 in range(0, T, Q):
        sl = slice(c0, min(c0 + Q, T))
        dtc, xc, Bc, Cc = dt[sl], x[sl], B[sl], C[sl]
        cs = np.cumsum(dtc * A)  # step 1: chunk cumsum
        CB = Cc @ Bc.T  # step 2: BMM
        w = np.exp(cs[-1] - cs) * dtc  # step 3: chunk state
        s = (w[:, None] * xc).T @ Bc
        Lm = np.exp(segsum(dtc * A))  # step 5: chunk scan
        y[sl] = (Lm * CB) @ (dtc[:, None] * xc) + np.exp(cs)[:, None] * (Cc @ S.T) + D * xc
        S = np.exp(cs[-1]) * S + s  # step 4: state passing
    return y, S


def linear_attention(x, dt, B, C, D, h0):
    """A = 0 closed form: no decay, the state is a running sum (linear attention)."""
    upd = dt[:, None, None] * x[:, :, None] * B[:, None, :]  # [T, P, N]
    hs = h0[None] + np.cumsum(upd, axis=0)
    y = np.einsum("tn,tpn->tp", C, hs) + D * x
    return y, (hs[-1] if len(dt) else h0.copy())
