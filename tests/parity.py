"""Parity gates between the CUDA path and the CPU oracle.

Tolerances (the bars the GPU path is held to):
  fp32 I/O:       max |y - y_ref| <= 1e-3 * RMS(y_ref)           (and the same for final states)
  bf16/fp16 I/O:  |y - y_ref| <= 1e-2 + r * |y_ref| element-wise, r = 2^-8 (bf16) or 2^-10 (fp16):
                  absolute 1e-2 on the value, plus one rounding of the stored output to its
                  16-bit type (a bf16 y of magnitude 16 cannot be within 1e-2 of anything).
  final states:   the same rule with r for the state dtype (0 for fp32 states) on top of the
                  I/O rounding term.
  fp16 states:    the state is stored in 16 bits wherever it is passed (every chunk), so the
                  fp32 gate applies only when both the I/O and the states are fp32. fp32 I/O
                  with fp16 states takes the 16-bit rule with r = 2^-10 (the passed state's
                  rounding).
  tensor-core path (16-bit I/O): its contractions take fp16 operands (P, X_s, S_in rounded
                  to 11 significant bits, the fused kernel's relaxed intermediates of the
                  kernel-fusion page's precision section), so one dominant product of y carries
                  up to two operand roundings, 2 * 2^-11 = 2^-10 of |y|, on top of the output's
                  own rounding: r = r(I/O) + 2^-10 whatever the state dtype. The plain rule
                  (r = r(I/O)) leaves only the fixed 1e-2 for that error where |y| sits just above
                  a power of two (a bf16 y of 130 rounds by up to 0.5 = 2^-8 * 128), which a
                  single fp16-rounded product of |y| > ~20 can exceed; the fraction of elements
                  that also meet the plain rule is reported beside the gate ("plain_ok").
Tensor-core operand envelope (gate_y_tc_envelope), used only for inputs far outside the pages'
workload distributions (|y| in the hundreds, states >> 10): the tensor-core path rounds P, X_s
and S_in to fp16 before its contractions, so on top of the bf16 output rounding its error grows
with the magnitudes summed. Bound: 1e-2 + (2^-8 + 2^-10)|y_ref| + 2^-9 RMS_head(y_ref), i.e. the
gate above, plus the fp16 rounding of a dominant product (two operands, 2^-11 each), plus about
five standard deviations of the rounding noise of an N-term fp16 contraction (2^-11/sqrt(3)
relative per term, summing to about 2^-12 of the per-head output scale).
The match percentages at tolerance 0 / 1e-3 / 1e-2 are reported beside the gate,
in the format of the fused-kernel page's precision table.
"""
from __future__ import annotations

import numpy as np

REL = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -10}


def stats(got, ref):
    d = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    return {
        "max_abs": float(d.max()) if d.size else 0.0,
        "rms_ref": rms,
        "max_over_rms": float(d.max() / rms) if d.size and rms > 0 else 0.0,
        "match_0": float(np.mean(d == 0)) if d.size else 1.0,
        "match_1e-3": float(np.mean(d <= 1e-3)) if d.size else 1.0,
        "match_1e-2": float(np.mean(d <= 1e-2)) if d.size else 1.0,
    }


TC_OPERAND = 2.0 ** -10  # two fp16 operand roundings of a dominant product (tensor-core path)


def gate_y(got, ref, io: str, state: str = "f32", tc: bool = False):
    """Return (ok, stats) for the output y (state: the dtype the states are passed in; tc: computed by the
    tensor-core path, whose contractions take fp16 operands)."""
    s = stats(got, ref)
    if got.size == 0:
        return True, s
    if io == "f32" and state == "f32":
        ok = s["max_abs"] <= 1e-3 * s["rms_ref"]
    else:
        r = REL[state] if io == "f32" else REL[io]
        err = np.abs(got - ref)
        plain = 1e-2 + r * np.abs(ref)
        s["plain_ok"] = float(np.mean(err <= plain))
        s["plain_worst_margin"] = float((err - plain).max())
        bound = plain + (TC_OPERAND * np.abs(ref) if tc and io != "f32" else 0.0)
        excess = err - bound
        s["worst_margin"] = float(excess.max())
        ok = bool(np.all(excess <= 0))
    return ok, s


def gate_final(got, ref, io: str, state: str):
    s = stats(got, ref)
    if got.size == 0:
        return True, s
    if io == "f32" and state == "f32":
        ok = s["max_abs"] <= 1e-3 * max(s["rms_ref"], 1e-30)
    else:
        bound = 1e-2 + (REL[state] + REL[io]) * np.abs(ref)
        ok = bool(np.all(np.abs(got - ref) <= bound))
    return ok, s


def gate_y_tc_envelope(got, ref, head_axis=2):
    """(ok, stats) under the tensor-core operand envelope (16-bit I/O only)."""
    s = stats(got, ref)
    if got.size == 0:
        return True, s
    axes = tuple(a for a in range(ref.ndim) if a != head_axis)
    rms_h = np.sqrt(np.mean(ref ** 2, axis=axes, keepdims=True))
    bound = 1e-2 + (2.0 ** -8 + 2.0 ** -10) * np.abs(ref) + 2.0 ** -9 * rms_h
    excess = np.abs(got - ref) - bound
    s["worst_margin"] = float(excess.max())
    return bool(np.all(excess <= 0)), s
