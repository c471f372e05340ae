"""Pins for the CPU oracle (no GPU needed).

Each check takes an implementation ``impl(x, dt_raw, dt_bias, A, B, C, D, h0)``
working on one chain in float64 (x [T, P], dt_raw [T], B/C [T, N], h0 [P, N];
dt_bias, A, D scalars) and returning (y [T, P], final [P, N]). The tests run
every check on the oracle; ``test_pins_catch_planted_mistakes`` runs them on
deliberately broken CPU recurrences to show each plausible mistake is caught.
"""
import json
import os

import numpy as np
import pytest

import oracle
import ssd_pins as pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def oracle_impl(x, dt_raw, dt_bias, A, B, C, D, h0):
    y, f = oracle.ssd_chains(x[None], dt_raw[None], np.array([dt_bias]), np.array([A]), B[None], C[None],
                             np.array([D]), h0[None], nthreads=1)
    return y[0], f[0]


def rand_chain(rng, T, P, N, dt_scale=1.0, init_scale=0.3):
    x = rng.standard_normal((T, P))
    dt_raw = rng.standard_normal(T) * dt_scale
    dt_bias = float(rng.uniform(-3.0, 0.5))
    A = -float(np.exp(rng.uniform(0.0, np.log(16.0))))
    B = rng.standard_normal((T, N))
    C = rng.standard_normal((T, N))
    D = float(rng.standard_normal())
    h0 = rng.standard_normal((P, N)) * init_scale
    return x, dt_raw, dt_bias, A, B, C, D, h0


def close(a, b, rtol=1e-11):
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= rtol * scale, f"max abs err {err:.3e} > {rtol:.1e} * {scale:.3e}"


# ---------------------------------------------------------------- checks
def check_golden(impl):
    for name in ("two_token_p1n1.json", "two_token_p2n3.json"):
        g = json.load(open(os.path.join(GOLDEN, name)))
        y, f = impl(np.array(g["x"], float), np.array(g["dt_raw"], float), g["dt_bias"], g["A"],
                    np.array(g["B"], float), np.array(g["C"], float), g["D"], np.array(g["init"], float))
        close(y, np.array(g["y"]), 1e-12)
        close(f, np.array(g["final"]), 1e-12)


def check_quadratic(impl, seed=1):
    rng = np.random.default_rng(seed)
    for T, P, N in ((1, 3, 2), (17, 4, 5), (64, 8, 16)):
        x, dtr, bias, A, B, C, D, h0 = rand_chain(rng, T, P, N)
        y, f = impl(x, dtr, bias, A, B, C, D, h0)
        yq, fq = pins.quadratic(x, pins.softplus(dtr + bias), A, B, C, D, h0)
        close(y, yq, 1e-11)
        close(f, fq, 1e-11)


def check_chunked_every_q(impl, seed=2):
    rng = np.random.default_rng(seed)
    T, P, N = 37, 3, 4
    x, dtr, bias, A, B, C, D, h0 = rand_chain(rng, T, P, N)
    y, f = impl(x, dtr, bias, A, B, C, D, h0)
    dt = pins.softplus(dtr + bias)
    for Q in range(1, T + 1):
        yc, fc = pins.chunked(x, dt, A, B, C, D, h0, Q)
        close(y, yc, 1e-11)
        close(f, fc, 1e-11)


def check_dt_zero(impl, seed=3):
    rng = np.random.default_rng(seed)
    x, dtr, _, A, B, C, D, h0 = rand_chain(rng, 23, 3, 5)
    y, f = impl(x, dtr, -1.0e4, A, B, C, D, h0)  # softplus(-1e4) == 0 exactly in fp64
    close(y, C @ h0.T + D * x, 1e-13)
    close(f, h0, 1e-13)


def check_linear_attention(impl, seed=4):
    rng = np.random.default_rng(seed)
    x, dtr, bias, _, B, C, D, h0 = rand_chain(rng, 29, 4, 3)
    y, f = impl(x, dtr, bias, 0.0, B, C, D, h0)
    yl, fl = pins.linear_attention(x, pins.softplus(dtr + bias), B, C, D, h0)
    close(y, yl, 1e-11)
    close(f, fl, 1e-11)


def check_split_rerun(impl, seed=5):
    rng = np.random.default_rng(seed)
    x, dtr, bias, A, B, C, D, h0 = rand_chain(rng, 50, 3, 4)
    y, f = impl(x, dtr, bias, A, B, C, D, h0)
    for T1 in (1, 16, 23, 49):
        y1, s = impl(x[:T1], dtr[:T1], bias, A, B[:T1], C[:T1], D, h0)
        y2, f2 = impl(x[T1:], dtr[T1:], bias, A, B[T1:], C[T1:], D, s)
        close(np.concatenate([y1, y2]), y, 1e-12)
        close(f2, f, 1e-12)


def check_linearity(impl, seed=6):
    rng = np.random.default_rng(seed)
    xa, dtr, bias, A, B, C, D, ha = rand_chain(rng, 31, 3, 4)
    xb = rng.standard_normal(xa.shape)
    hb = rng.standard_normal(ha.shape)
    ya, fa = impl(xa, dtr, bias, A, B, C, D, ha)
    yb, fb = impl(xb, dtr, bias, A, B, C, D, hb)
    ys, fs = impl(2.0 * xa - xb, dtr, bias, A, B, C, D, 2.0 * ha - hb)
    close(ys, 2.0 * ya - yb, 1e-11)
    close(fs, 2.0 * fa - fb, 1e-11)


def check_b_zero(impl, seed=7):
    rng = np.random.default_rng(seed)
    x, dtr, bias, A, _, C, D, h0 = rand_chain(rng, 19, 3, 4)
    B = np.zeros((19, 4))
    y, f = impl(x, dtr, bias, A, B, C, D, h0)
    cs = np.cumsum(pins.softplus(dtr + bias) * A)
    close(y, np.exp(cs)[:, None] * (C @ h0.T) + D * x, 1e-12)
    close(f, np.exp(cs[-1]) * h0, 1e-12)


CHECKS = [check_golden, check_quadratic, check_chunked_every_q, check_dt_zero, check_linear_attention,
          check_split_rerun, check_linearity, check_b_zero]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle_impl)


# ---------------------------------------------------------------- multi-chain wrapper
def test_reference_layout_and_groups():
    """ssd_reference gathers chains with g = h // (H/G); heads/batches are independent."""
    rng = np.random.default_rng(11)
    b, L, H, P, N, G = 2, 13, 4, 3, 5, 2
    x = rng.standard_normal((b, L, H, P))
    dtr = rng.standard_normal((b, L, H))
    bias = rng.uniform(-3, 0, H)
    A = -np.exp(rng.uniform(0, 2.7, H))
    B = rng.standard_normal((b, L, G, N))
    C = rng.standard_normal((b, L, G, N))
    D = rng.standard_normal(H)
    h0 = rng.standard_normal((b, H, P, N))
    y, f = oracle.ssd_reference(x, dtr, bias, A, B, C, D, h0, nthreads=3)
    for bi in range(b):
        for h in range(H):
            g = h // (H // G)
            yc, fc = pins.quadratic(x[bi, :, h], pins.softplus(dtr[bi, :, h] + bias[h]), A[h], B[bi, :, g],
                                    C[bi, :, g], D[h], h0[bi, h])
            close(y[bi, :, h], yc, 1e-11)
            close(f[bi, h], fc, 1e-11)
    ys, fs = oracle.ssd_reference(x, dtr, bias, A, B, C, D, h0, chains=[(1, 3), (0, 0)])
    close(ys[0], y[1, :, 3], 0)
    close(fs[1], f[0, 0], 0)
    # no D and no init state mean zero
    y0, f0 = oracle.ssd_reference(x, dtr, bias, A, B, C, None, None)
    y1, f1 = oracle.ssd_reference(x, dtr, bias, A, B, C, np.zeros(H), np.zeros_like(h0))
    close(y0, y1, 0)
    close(f0, f1, 0)


def test_empty_sequence():
    x = np.zeros((1, 0, 2, 4))
    y, f = oracle.ssd_reference(x, np.zeros((1, 0, 2)), np.zeros(2), -np.ones(2), np.zeros((1, 0, 1, 3)),
                                np.zeros((1, 0, 1, 3)), None, np.ones((1, 2, 4, 3)))
    assert y.shape == (1, 0, 2, 4)
    assert np.array_equal(f, np.ones((1, 2, 4, 3)))


# ---------------------------------------------------------------- planted mistakes
def _mutant(kind):
    """A pure-Python recurrence with one planted mistake (CPU only)."""

    def impl(x, dt_raw, dt_bias, A, B, C, D, h0):
        T, P = x.shape
        N = B.shape[1]
        h = h0.copy()
        y = np.zeros((T, P))
        for t in range(T):
            v = dt_raw[t] + dt_bias
            dt = v if kind == "no_softplus" else float(pins.softplus(v))
            a = dt * (-A if kind == "decay_sign" else A)
            decay = np.exp(a)
            if kind == "zoh_b":  # exact ZOH input matrix instead of dt*B
                bt = (np.expm1(a) / A if A != 0 else dt) * B[t]
            elif kind == "b_for_c":
                bt = dt * C[t]
            else:
                bt = dt * B[t]
            if kind == "transposed":
                h = decay * h + np.outer(x[t], bt[::-1])
            elif kind == "late_decay":  # decay applied after the update
                h = decay * (h + np.outer(x[t], bt))
            else:
                h = decay * h + np.outer(x[t], bt)
            prev = h if kind != "y_before_update" else (h - np.outer(x[t], bt))
            y[t] = prev @ C[t] + (0.0 if kind == "no_d" else D) * x[t]
        return y, h

    return impl


MUTANTS = ["no_softplus", "decay_sign", "zoh_b", "b_for_c", "transposed", "late_decay", "y_before_update", "no_d"]


def test_pins_accept_a_correct_python_recurrence():
    good = _mutant("none")
    for check in CHECKS:
        check(good)


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistakes(kind):
    bad = _mutant(kind)
    failed = []
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(bad)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {kind!r}"


def test_varlen_oracle_against_the_worked_examples():
    """Variable-length packing: the worked two-token examples packed twice around an empty sequence along one
    token axis must give each example's hand-derived y and final state, and the empty sequence keeps its
    initial state (each sequence restarts the recurrence from its own initial state)."""
    for name in ("two_token_p1n1.json", "two_token_p2n3.json"):
        g = json.load(open(os.path.join(GOLDEN, name)))
        x, dtr = np.array(g["x"], float), np.array(g["dt_raw"], float)
        B, C, h0 = np.array(g["B"], float), np.array(g["C"], float), np.array(g["init"], float)
        P, N = h0.shape
        xx = np.concatenate([x, x])[None, :, None, :]
        dd = np.concatenate([dtr, dtr])[None, :, None]
        BB = np.concatenate([B, B])[None, :, None, :]
        CC = np.concatenate([C, C])[None, :, None, :]
        empty_init = np.full((P, N), 7.0)
        init = np.stack([h0, empty_init, h0])[:, None]
        y, f = oracle.ssd_varlen_reference(xx, dd, np.array([g["dt_bias"]]), np.array([g["A"]]), BB, CC,
                                           np.array([0, 2, 2, 4]), np.array([g["D"]]), init)
        for half in (0, 1):
            close(y[0, 2 * half:2 * half + 2, 0], np.array(g["y"]), 1e-12)
        close(f[0, 0], np.array(g["final"]), 1e-12)
        close(f[2, 0], np.array(g["final"]), 1e-12)
        close(f[1, 0], empty_init, 0.0)


def test_conv_oracle_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "conv_k3_two_channels.json")))
    out, st = oracle.conv1d_reference(np.array(g["xbc"]), np.array(g["weight"]), np.array(g["bias"]),
                                      np.array(g["conv_state"]), activation="none")
    close(out, np.array(g["out"]), 1e-15)
    close(st, np.array(g["state_out"]), 0.0)


def test_conv_oracle_against_numpy_convolve_and_silu():
    """Every channel against numpy's full convolution (a library primitive) of [state, tokens] with the flipped
    taps, plus the closed-form SiLU v / (1 + e^-v); and a split sequence continued through the conv cache."""
    rng = np.random.default_rng(5)
    b, L, D, k = 2, 9, 5, 4
    x = rng.standard_normal((b, L, D))
    w = rng.standard_normal((D, k))
    bias = rng.standard_normal(D)
    st = rng.standard_normal((b, D, k - 1))
    out, st_out = oracle.conv1d_reference(x, w, bias, st, activation="silu")
    for bi in range(b):
        for ch in range(D):
            seq = np.concatenate([st[bi, ch], x[bi, :, ch]])
            ref = np.convolve(seq, w[ch, ::-1], mode="valid") + bias[ch]
            close(out[bi, :, ch], ref / (1.0 + np.exp(-ref)), 1e-13)
            close(st_out[bi, ch], x[bi, L - (k - 1):, ch], 0.0)
    o1, s1 = oracle.conv1d_reference(x[:, :4], w, bias, st)
    o2, s2 = oracle.conv1d_reference(x[:, 4:], w, bias, s1)
    close(np.concatenate([o1, o2], axis=1), out, 1e-15)
    close(s2, st_out, 0.0)


def test_conv_oracle_width_one_and_sequences_shorter_than_the_cache():
    """Width 1 (no history: a per-channel scale and bias, an empty cache) and widths up to 8 on sequences shorter
    than the cache (the cache leaving the sequence is then the tail of [cache on entry, tokens]), each against
    numpy's convolution of [cache, tokens] with the flipped taps."""
    rng = np.random.default_rng(11)
    b, D = 2, 3
    x = rng.standard_normal((b, 5, D))
    w1 = rng.standard_normal((D, 1))
    bias = rng.standard_normal(D)
    out, st = oracle.conv1d_reference(x, w1, bias, None, activation="none")
    close(out, x * w1[:, 0] + bias, 1e-15)
    assert st.shape == (b, D, 0)
    for k, L in ((6, 2), (8, 1), (8, 7), (5, 4)):
        xs = rng.standard_normal((b, L, D))
        w = rng.standard_normal((D, k))
        cache = rng.standard_normal((b, D, k - 1))
        out, st = oracle.conv1d_reference(xs, w, bias, cache, activation="none")
        for bi in range(b):
            for ch in range(D):
                seq = np.concatenate([cache[bi, ch], xs[bi, :, ch]])
                close(out[bi, :, ch], np.convolve(seq, w[ch, ::-1], mode="valid") + bias[ch], 1e-13)
                close(st[bi, ch], seq[-(k - 1):], 0.0)


def test_conv_ssd_oracle_channel_split_worked_example():
    """The x | B | C split of the convolved rows (x the first H*P channels, then B's G*N, then C's G*N): the
    hand-worked two-token example with P = 2, N = 3 (its B and C differ, so a swap of the two slices, or x read
    from the wrong channels, changes y) laid out as raw rows [x(2), B(3), C(3)] and passed through a width-1
    identity convolution must give the example's hand-derived y and final state."""
    g = json.load(open(os.path.join(GOLDEN, "two_token_p2n3.json")))
    x, B, C = np.array(g["x"]), np.array(g["B"]), np.array(g["C"])
    xbc = np.concatenate([x, B, C], axis=1)[None]  # [1, 2, 8]
    ident = np.ones((8, 1))
    y, f, st = oracle.ssd_conv_reference(xbc, ident, None, np.array(g["dt_raw"])[None, :, None],
                                         np.array([g["dt_bias"]]), np.array([g["A"]]), nheads=1, headdim=2,
                                         ngroups=1, dstate=3, D=np.array([g["D"]]),
                                         init_states=np.array(g["init"])[None, None], activation="none")
    close(y[0, :, 0], np.array(g["y"]), 1e-12)
    close(f[0, 0], np.array(g["final"]), 1e-12)
    assert st.shape == (1, 8, 0)


def test_conv_ssd_oracle_channel_split_heads_and_groups():
    """Three heads in three groups: the convolved rows sliced here channel by channel (x of head h, element p at
    channel h*P + p; B of group g, element n at H*P + g*N + n; C at H*P + G*N + g*N + n) and run through the plain
    oracle equal the conv oracle's own split."""
    rng = np.random.default_rng(5)
    b, L, H, P, G, N, k = 2, 9, 3, 2, 3, 4, 3
    Dc = H * P + 2 * G * N
    xbc = rng.standard_normal((b, L, Dc))
    w = rng.standard_normal((Dc, k))
    bias = rng.standard_normal(Dc)
    cache = rng.standard_normal((b, Dc, k - 1))
    dt_raw = rng.standard_normal((b, L, H))
    dt_bias, A, Dh = rng.standard_normal(H), -np.exp(rng.uniform(0, 2, H)), rng.standard_normal(H)
    init = rng.standard_normal((b, H, P, N)) * 0.3
    y, f, _ = oracle.ssd_conv_reference(xbc, w, bias, dt_raw, dt_bias, A, nheads=H, headdim=P, ngroups=G, dstate=N,
                                        D=Dh, init_states=init, conv_state=cache, activation="silu")
    out, _ = oracle.conv1d_reference(xbc, w, bias, cache, "silu")
    xs = np.empty((b, L, H, P))
    Bs = np.empty((b, L, G, N))
    Cs = np.empty((b, L, G, N))
    for h in range(H):
        for p in range(P):
            xs[:, :, h, p] = out[:, :, h * P + p]
    for gg in range(G):
        for n in range(N):
            Bs[:, :, gg, n] = out[:, :, H * P + gg * N + n]
            Cs[:, :, gg, n] = out[:, :, H * P + G * N + gg * N + n]
    yr, fr = oracle.ssd_reference(xs, dt_raw, dt_bias, A, Bs, Cs, Dh, init)
    close(y, yr, 1e-13)
    close(f, fr, 1e-13)
