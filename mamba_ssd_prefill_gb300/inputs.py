"""Seeded synthetic inputs for the SSD prefill forward.

This module only draws random numbers; it holds none of the SSD arithmetic,
so both the CUDA path's tests and the CPU oracle can use it.

Workload shapes follow the Mamba-2 layer shapes the benchmarks of "Accelerating
Mamba2 with Kernel Fusion" sweep (batch 1-32, sequence 1K-256K, fp16 states,
the 130M and 2.7B models): headdim 64, d_state 128, 24 or 80 heads.

Value recipe (per tensor):
  x, B, C, dt_raw ~ N(0, 1), cast to the I/O dtype
  dt_bias[h]      = inverse-softplus(dt0_h), dt0_h log-uniform in [dt_lo, 0.1]
  A[h]            = -exp(U[log 1, log 16])
  D[h]            ~ N(0, 1)
  init_states     zeros, absent, or N(0, 0.1^2) in the state dtype
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    io: str = "bf16"  # x, dt_raw, B, C, y
    state: str = "f32"  # init/final and passed states
    init: str = "normal"  # "zeros" | "none" | "normal"
    dt_lo: float = 1e-3
    seed: int = 0

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workload families (sizes as named); seeds are fixed per family.
WORKLOADS = {
    "tiny-fp32": Workload("tiny-fp32", 1, 1024, 8, 64, 64, 1, 128, io="f32", state="f32", init="zeros", seed=1001),
    "m130-bf16": Workload("m130-bf16", 4, 4096, 24, 64, 128, 1, 128, io="bf16", state="f32", init="normal", seed=1002),
    "m2p7-L16k-q128": Workload("m2p7-L16k-q128", 1, 16384, 80, 64, 128, 1, 128, io="bf16", state="f16", init="none", seed=1003),
    "m2p7-L16k-q256": Workload("m2p7-L16k-q256", 1, 16384, 80, 64, 128, 1, 256, io="bf16", state="f16", init="none", seed=1003),
    "m2p7-L8k-b1": Workload("m2p7-L8k-b1", 1, 8192, 80, 64, 128, 1, 128, io="bf16", state="f32", init="normal", seed=1004),
    "m2p7-L8k-b8": Workload("m2p7-L8k-b8", 8, 8192, 80, 64, 128, 1, 128, io="bf16", state="f32", init="normal", seed=1004),
    "m2p7-L8k-b32": Workload("m2p7-L8k-b32", 32, 8192, 80, 64, 128, 1, 128, io="bf16", state="f32", init="normal", seed=1004),
    "m2p7-L8k-b8-f16": Workload("m2p7-L8k-b8-f16", 8, 8192, 80, 64, 128, 1, 128, io="bf16", state="f16", init="normal",
                                seed=1004),
    "long-L256k-g8": Workload("long-L256k-g8", 1, 262144, 80, 64, 128, 8, 128, io="bf16", state="f32", init="none",
                              dt_lo=1e-4, seed=1005),
    # the long-context layer at 1/8 of its length (profiling captures: 0.8 GB of inputs and outputs)
    "long-L32k-g8": Workload("long-L32k-g8", 1, 32768, 80, 64, 128, 8, 128, io="bf16", state="f32", init="none",
                             dt_lo=1e-4, seed=1005),
    # the fp16-state variants of the fp32-state workloads above (states passed and returned in fp16)
    "long-L256k-g8-f16": Workload("long-L256k-g8-f16", 1, 262144, 80, 64, 128, 8, 128, io="bf16", state="f16",
                                  init="none", dt_lo=1e-4, seed=1005),
    "m130-bf16-f16": Workload("m130-bf16-f16", 4, 4096, 24, 64, 128, 1, 128, io="bf16", state="f16", init="normal",
                              seed=1002),
    # decode: one token per sequence advances the cached state (2.7B layer shape, 64 / 256 sequences)
    "decode-2p7-b64": Workload("decode-2p7-b64", 64, 1, 80, 64, 128, 1, 128, io="bf16", state="f32", init="normal",
                               seed=1006),
    "decode-2p7-b256-f16": Workload("decode-2p7-b256-f16", 256, 1, 80, 64, 128, 1, 128, io="bf16", state="f16",
                                    init="normal", seed=1007),
}


def make_inputs(w: Workload, device="cpu", seed: int | None = None) -> dict:
    """Draw one seeded input set for workload ``w`` on ``device``.

    Returns a dict with x, dt_raw, dt_bias, A, B, C, D, init_states (None when
    the workload has no init state). Per-head parameters are drawn on the CPU
    so they do not depend on the device; the large tensors use a generator on
    ``device``.
    """
    seed = w.seed if seed is None else seed
    io = DTYPES[w.io]
    st = DTYPES[w.state]
    b, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    gcpu = torch.Generator("cpu").manual_seed(seed)
    dt0 = torch.exp(torch.empty(H, dtype=torch.float64).uniform_(math.log(w.dt_lo), math.log(0.1), generator=gcpu))
    dt_bias = torch.log(torch.expm1(dt0)).to(torch.float32)  # inverse of softplus
    A = (-torch.exp(torch.empty(H, dtype=torch.float64).uniform_(0.0, math.log(16.0), generator=gcpu))).to(torch.float32)
    D = torch.randn(H, generator=gcpu, dtype=torch.float32)
    g = torch.Generator(device).manual_seed(seed + 1)

    def randn(*shape, scale=1.0, dtype=io):
        t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        if scale != 1.0:
            t.mul_(scale)
        return t.to(dtype)

    x = randn(b, L, H, P)
    dt_raw = randn(b, L, H)
    B = randn(b, L, G, N)
    C = randn(b, L, G, N)
    if w.init == "normal":
        init = randn(b, H, P, N, scale=0.1, dtype=st)
    elif w.init == "zeros":
        init = torch.zeros(b, H, P, N, device=device, dtype=st)
    else:
        init = None
    return dict(x=x, dt_raw=dt_raw, dt_bias=dt_bias.to(device), A=A.to(device), B=B, C=C, D=D.to(device),
                init_states=init)


def make_varlen_inputs(w: Workload, lengths, device="cpu", seed: int | None = None) -> dict:
    """A variable-length batch with the shapes and distributions of ``w``: the sequences of ``lengths`` packed
    along one token axis ([1, T, ...] tensors, T = sum of lengths), cu_seqlens (int32 [nseq + 1]) and, when the
    workload has an initial state, init_states [nseq, H, P, N]."""
    seed = w.seed if seed is None else seed
    T = int(sum(lengths))
    inp = make_inputs(w.with_(batch=1, seqlen=T, init="none"), device=device, seed=seed)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(list(lengths), dtype=torch.int64), 0).to(torch.int32)
    inp["cu_seqlens"] = cu.to(device)
    if w.init != "none":
        g = torch.Generator(device).manual_seed(seed + 2)
        st = torch.randn(len(lengths), w.nheads, w.headdim, w.dstate, generator=g, device=device)
        inp["init_states"] = (st.mul_(0.1) if w.init == "normal" else st.zero_()).to(DTYPES[w.state])
    return inp


def make_conv_inputs(w: Workload, width: int = 4, device="cpu", seed: int | None = None, conv_state: bool = True) -> dict:
    """Raw inputs of the convolution in front of the SSD, with the SSD parameters of ``w``: xbc [b, L, H*P + 2*G*N]
    ~ N(0, 1) in the I/O dtype, conv taps ~ U(-1, 1) / sqrt(width), bias ~ N(0, 0.1^2), and (optionally) a conv
    cache [b, D, width - 1] ~ N(0, 1)."""
    seed = w.seed if seed is None else seed
    inp = make_inputs(w, device=device, seed=seed)
    D = w.nheads * w.headdim + 2 * w.ngroups * w.dstate
    g = torch.Generator(device).manual_seed(seed + 3)
    out = dict(dt_raw=inp["dt_raw"], dt_bias=inp["dt_bias"], A=inp["A"], D=inp["D"], init_states=inp["init_states"])
    out["xbc"] = torch.randn(w.batch, w.seqlen, D, generator=g, device=device).to(DTYPES[w.io])
    out["conv_weight"] = ((torch.rand(D, width, generator=g, device=device) * 2 - 1) / math.sqrt(width)).contiguous()
    out["conv_bias"] = torch.randn(D, generator=g, device=device) * 0.1
    out["conv_state"] = (torch.randn(w.batch, D, width - 1, generator=g, device=device).to(DTYPES[w.io])
                         if conv_state and width > 1 else None)
    return out


def make_chain_inputs(w: Workload, n: int, seed: int | None = None) -> dict:
    """n independent (sequence, head) chains of workload ``w`` drawn directly on the CPU in float64, with the value
    recipe above, for timing the oracle on a bounded sample without materialising the whole batch: x [n, L, P],
    dt_raw [n, L], B/C [n, L, N] (the B and C columns of each chain's group), dt_bias/A/D [n] (each chain's head
    drawn from the per-head recipe), init [n, P, N] or None. The numbers are not those of ``make_inputs`` (a
    different generator layout); the shapes and distributions are."""
    import numpy as np

    seed = w.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    L, P, N = w.seqlen, w.headdim, w.dstate
    dt0 = np.exp(rng.uniform(math.log(w.dt_lo), math.log(0.1), n))
    out = dict(x=rng.standard_normal((n, L, P)), dt_raw=rng.standard_normal((n, L)),
               dt_bias=np.log(np.expm1(dt0)), A=-np.exp(rng.uniform(0.0, math.log(16.0), n)),
               B=rng.standard_normal((n, L, N)), C=rng.standard_normal((n, L, N)), D=rng.standard_normal(n))
    out["init"] = rng.standard_normal((n, P, N)) * 0.1 if w.init == "normal" else (
        np.zeros((n, P, N)) if w.init == "zeros" else None)
    return out
