"""Pins for the CPU oracle: each check ties it to something other than itself.

Closed forms, a library routine (torch's float32 -> bfloat16 rounding), an independent
high-precision brute force (mpmath at 200 bits), and invariants the pages fix. The
`planted` tests substitute a plausible mistake into the oracle (on the CPU) and show
that one of the pins catches it.
"""
import math

import mpmath
import numpy as np
import pytest
import torch

from oracle import ga_oracle as O
from verify_gated_gqa_gb300 import synth

mpmath.mp.prec = 200


# ---------------------------------------------------------------- bf16 rounding
def test_bf16_matches_torch_rne():
    """Library routine: torch rounds float32 -> bfloat16 to nearest even."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal(200000).astype(np.float32)
    x = np.concatenate([x, (x * np.float32(1e-38)), (x * np.float32(1e30)),
                        np.float32([3.3e38, -3.3e38, 0.0, -0.0])]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    got = O.bf16(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_ties_and_overflow():
    assert O.bf16(1 + 2.0 ** -8) == 1.0                       # tie -> even (down)
    assert O.bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6          # tie -> even (up)
    assert O.bf16(-(1 + 3 * 2.0 ** -8)) == -(1 + 2.0 ** -6)
    assert O.bf16(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7  # just above the tie
    assert np.isinf(O.bf16(3.4e38))
    assert O.bf16(2.0 ** -133) == 2.0 ** -133                  # smallest subnormal
    # double rounding through float32 would give a different answer here:
    x = 1 + 2.0 ** -8 + 2.0 ** -40   # float32(x) is the tie 1 + 2^-8 -> 1.0
    assert O.bf16(x) == 1 + 2.0 ** -7


def test_bf16_sig_unbounded_exponent():
    x = 2.0 ** -140 * (1 + 2.0 ** -7 + 2.0 ** -12)
    assert O.bf16_sig(x) == 2.0 ** -140 * (1 + 2.0 ** -7)
    x = np.random.default_rng(2).standard_normal(1000) * 10
    assert np.array_equal(O.bf16_sig(x), O.bf16(x))


def test_ulp_closed_forms():
    assert O.ulp_bf16(1.0) == 2.0 ** -7
    assert O.ulp_bf16(1.99) == 2.0 ** -7
    assert O.ulp_bf16(2.0) == 2.0 ** -6
    assert O.ulp_bf16(0.0018157959) == 2.0 ** -17
    assert O.ulp_bf16(-3.0) == 2.0 ** -6


# ---------------------------------------------------------------- RoPE table
def test_rope_table_position_zero_and_frequencies():
    c, s = O.rope_tables(70000, rounded=False)
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
    # angle of pair i at position 1 is 10^(-7 i / 32) (closed form of 1e7^(-2i/64))
    theta = np.arctan2(s[1], c[1])
    want = np.array([10.0 ** (-7.0 * i / 32.0) for i in range(32)])
    assert np.allclose(theta, want, rtol=1e-12, atol=0)
    # the angle grows linearly in the position (pair 31 never wraps before 70000)
    p = np.array([1, 777, 65551])
    assert np.allclose(np.arctan2(s[p, 31], c[p, 31]), p * want[31], rtol=1e-10)
    assert np.allclose(c ** 2 + s ** 2, 1.0, atol=1e-15)


def test_rope_table_rounded_once():
    cu, su = O.rope_tables(4096, rounded=False)
    cr, sr = O.rope_tables(4096, rounded=True)
    assert np.array_equal(cr, O.bf16(cu)) and np.array_equal(sr, O.bf16(su))
    # against mpmath at 200 bits, rounded once to bf16 with Python's own float rounding
    for p, i in [(1, 0), (2054, 5), (4095, 31), (3000, 17)]:
        ang = mpmath.mpf(p) * mpmath.power(mpmath.mpf(10) ** 7, -mpmath.mpf(2 * i) / 64)
        want_c = _rne_bf16_mp(mpmath.cos(ang))
        want_s = _rne_bf16_mp(mpmath.sin(ang))
        assert cr[p, i] == want_c and sr[p, i] == want_s


def _rne_bf16_mp(x):
    """Independent RNE to bf16 from an mpmath value (exact rational arithmetic)."""
    from fractions import Fraction
    if x == 0:
        return 0.0
    f = Fraction(int(mpmath.floor(x * 2 ** 300)), 2 ** 300) if x > 0 else \
        -Fraction(int(mpmath.floor(-x * 2 ** 300)), 2 ** 300)
    sign = 1 if f > 0 else -1
    a = abs(f)
    e = math.floor(math.log2(float(a))) if float(a) > 0 else -200
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (max(e, -126) - 7)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * float(fl * q)


# ---------------------------------------------------------------- (1+w) RMSNorm
def test_norm_constant_vector_closed_form():
    for c in [1.0, -3.0, 0.015625, 40.0, 2.0 ** -10]:
        for w in [0.0, 0.5, -0.25]:
            x = np.full(256, c)
            want = O.bf16(np.sign(c) * (1 + w) / math.sqrt(1 + O.EPS / (c * c)))
            assert np.all(O.rms_norm_1pw(x, np.full(256, w)) == want)
    assert np.all(O.rms_norm_1pw(np.zeros(256), np.zeros(256)) == 0.0)


def test_norm_against_mpmath():
    rng = np.random.default_rng(3)
    x = O.bf16(rng.standard_normal((4, 256)))
    w = O.bf16(0.1 * rng.standard_normal(256))
    got = O.rms_norm_1pw(x, w)
    for r in range(4):
        ms = mpmath.fsum([mpmath.mpf(float(v)) ** 2 for v in x[r]]) / 256
        inv = 1 / mpmath.sqrt(ms + mpmath.mpf(O.EPS))
        for d in range(256):
            want = _rne_bf16_mp(mpmath.mpf(float(x[r, d])) * inv * (1 + mpmath.mpf(float(w[d]))))
            assert got[r, d] == want


def test_norm_scale_invariance_without_eps():
    x = O.bf16(np.random.default_rng(4).standard_normal(256))
    w = np.zeros(256)
    assert np.array_equal(O.rms_norm_1pw(4 * x, w, eps=0.0), O.rms_norm_1pw(x, w, eps=0.0))


# ---------------------------------------------------------------- partial RoPE
def test_rope_pairing_closed_form():
    """A unit vector on dim i (i < 32) rotates into dims i and i+32 by angle i."""
    c, s = O.rope_tables(100, rounded=False)
    p = 37
    for i in [0, 9, 31]:
        x = np.zeros(256)
        x[i] = 1.0
        y = O.rope_partial(x, c[p], s[p], rounded=False)
        want = np.zeros(256)
        want[i], want[i + 32] = c[p, i], s[p, i]
        assert np.array_equal(y, want)
    x = np.zeros(256)
    x[100] = 2.0
    assert np.array_equal(O.rope_partial(x, c[p], s[p]), x)     # dims >= 64 pass through


def test_rope_identity_norm_and_inverse():
    rng = np.random.default_rng(5)
    x = O.bf16(rng.standard_normal((3, 256)))
    cr, sr = O.rope_tables(9000)
    assert np.array_equal(O.rope_partial(x, cr[0], sr[0]), x)     # position 0 is the identity
    c, s = O.rope_tables(9000, rounded=False)
    p = 8191
    y = O.rope_partial(x, c[p], s[p], rounded=False)
    pair = lambda z: z[:, :32] ** 2 + z[:, 32:64] ** 2
    assert np.allclose(pair(y), pair(x), rtol=1e-13)
    back = O.rope_partial(y, c[p], -s[p], rounded=False)         # rotate by -angle
    assert np.allclose(back, x, atol=1e-12)


def test_rope_rounding_points_hand_worked():
    """[QSA], the attention-reader commit: cos/sin are bf16 and the rotation rounds in
    bf16, each product and then the sum. Hand-worked values where that differs from one
    rounding of the exact a*c - b*s (and of b*c + a*s):

    pair 0: a = 1 + 2^-6, b = -2^-9, c = 1 - 2^-8, s = 2^-4.
      a*c = 1 + 3*2^-8 - 2^-14, just below the midpoint 1 + 3*2^-8 of 1 + 2^-7 and
      1 + 2^-6, so bf16(a*c) = 1 + 2^-7; bf16(b*s) = -2^-13 (exact);
      bf16(1 + 2^-7 + 2^-13) = 1 + 2^-7.  One rounding of the exact value
      1 + 3*2^-8 + 2^-14 (above the midpoint) would give 1 + 2^-6.
      y_32 = bf16(bf16(b*c) + bf16(a*s)) = bf16(-(2^-9 - 2^-17) + (2^-4 + 2^-10))
           = 252 * 2^-12 (the step there is 2^-12).
    pair 1 mirrors it in the second formula: a = 2^-9, b = 1 + 2^-6:
      y_33 = bf16(bf16(b*c) + bf16(a*s)) = 1 + 2^-7 (one rounding: 1 + 2^-6),
      y_1 = -252 * 2^-12."""
    x = np.zeros(256)
    cos_row, sin_row = np.ones(32), np.zeros(32)
    x[0], x[32] = 1 + 2.0 ** -6, -(2.0 ** -9)
    x[1], x[33] = 2.0 ** -9, 1 + 2.0 ** -6
    cos_row[:2], sin_row[:2] = 1 - 2.0 ** -8, 2.0 ** -4
    x[2:32] = x[34:64] = 0.5
    x[100] = 3.0
    y = O.rope_partial(x, cos_row, sin_row)
    assert y[0] == 1 + 2.0 ** -7 and y[33] == 1 + 2.0 ** -7
    assert y[32] == 252 * 2.0 ** -12 and y[1] == -252 * 2.0 ** -12
    assert np.all(y[2:32] == 0.5) and np.all(y[34:64] == 0.5) and y[100] == 3.0
    # the single-rounding reading of the same pair, worked with exact rationals: the
    # values above are where the two readings part
    from fractions import Fraction as F
    exact = F(1) + F(1, 64) - F(1, 256) - F(1, 2 ** 14) + F(1, 2 ** 13)
    assert exact > F(1) + F(3, 256) and O.bf16(float(exact)) == 1 + 2.0 ** -6


# ---------------------------------------------------------------- brute force attention
def _mp_attention(qg, k, v, w_q, w_k, q_base, T, kind, mask=None, heads=(0, 12)):
    """Textbook gated GQA attention at 200 bits, written directly from the pages'
    description (no oracle code): split, (1+w) norm, partial RoPE at the exact angle,
    score q.k/16, softmax over visible keys, P.V, times sigmoid(gate)."""
    R = qg.shape[0]
    eps = mpmath.mpf(O.EPS)

    def norm(vec, w):
        vec = [mpmath.mpf(float(a)) for a in vec]
        ms = mpmath.fsum([a * a for a in vec]) / len(vec)
        inv = 1 / mpmath.sqrt(ms + eps)
        return [a * inv * (1 + mpmath.mpf(float(b))) for a, b in zip(vec, w)]

    def rope(vec, pos):
        out = list(vec)
        for i in range(32):
            ang = mpmath.mpf(pos) * mpmath.power(mpmath.mpf(10) ** 7, -mpmath.mpf(2 * i) / 64)
            cs, sn = mpmath.cos(ang), mpmath.sin(ang)
            out[i] = vec[i] * cs - vec[i + 32] * sn
            out[i + 32] = vec[i + 32] * cs + vec[i] * sn
        return out

    keys = {kv: [rope(norm(k[j, kv], w_k), j) for j in range(T)] for kv in (0, 1)}
    res = {}
    for h in heads:
        kv = h * 2 // 24
        for r in range(R):
            pos = q_base + r
            q = rope(norm(qg[r, h, :256], w_q), pos)
            vis = [j for j in range(T) if (j <= pos if kind == "causal" else
                                           (True if kind == "bidirectional" else mask[r, j] != 0))]
            sc = [mpmath.fsum([a * b for a, b in zip(q, keys[kv][j])]) / 16 for j in vis]
            m = max(sc)
            e = [mpmath.exp(x - m) for x in sc]
            z = mpmath.fsum(e)
            o = [mpmath.fsum([e[n] * mpmath.mpf(float(v[j, kv, d])) for n, j in enumerate(vis)]) / z
                 for d in range(256)]
            g = [1 / (1 + mpmath.exp(-mpmath.mpf(float(a)))) for a in qg[r, h, 256:]]
            res[(r, h)] = np.array([float(a * b) for a, b in zip(o, g)])
    return res


def _small_case(S=6, seed=11):
    qg, k, v, w_q, w_k = synth.attention_inputs(seed, S, S)
    f = lambda t: t.double().numpy()
    return f(qg), f(k), f(v), f(w_q), f(w_k)


@pytest.mark.parametrize("kind,q_base", [("causal", 0), ("bidirectional", 0), ("causal", 3)])
def test_f64_mode_equals_mp_bruteforce(kind, q_base):
    qg, k, v, w_q, w_k = _small_case(S=6)
    T = 6
    rows = qg[: T - q_base]
    ref = _mp_attention(rows, k, v, w_q, w_k, q_base, T, kind)
    c, s = O.rope_tables(T, rounded=False)
    kp = O.prep_keys(k, w_k, c, s, mode="F64")
    out = O.prefill(rows, kp, v, w_q, c, s, q_base, T, causal=(kind == "causal"), mode="F64")
    for (r, h), want in ref.items():
        assert np.allclose(out[r, h * 256:(h + 1) * 256], want, rtol=1e-12, atol=1e-14)


def test_r1_within_float64_bound_of_bruteforce():
    """[WIDE] review §Kernel change: the flash kernel is checked against a float64
    reference with a 1.6e-2 relative tolerance."""
    qg, k, v, w_q, w_k = _small_case(S=8, seed=12)
    ref = _mp_attention(qg, k, v, w_q, w_k, 0, 8, "causal")
    c, s = O.rope_tables(8)
    kp = O.prep_keys(k, w_k, c, s)
    out = O.prefill(qg, kp, v, w_q, c, s, 0, 8)
    for (r, h), want in ref.items():
        got = out[r, h * 256:(h + 1) * 256]
        assert np.linalg.norm(got - want) <= 1.6e-2 * np.linalg.norm(want)


def test_masked_f64_equals_mp_bruteforce():
    qg, k, v, w_q, w_k = _small_case(S=7, seed=13)
    mask = (np.random.default_rng(6).random((7, 7)) < 0.5).astype(np.uint8)
    mask[np.arange(7), np.arange(7)] = 1
    ref = _mp_attention(qg, k, v, w_q, w_k, 0, 7, "mask", mask)
    c, s = O.rope_tables(7, rounded=False)
    kp = O.prep_keys(k, w_k, c, s, mode="F64")
    out, _, _ = O.masked(qg, kp, v, w_q, c, s, 0, 7, mask, mode="F64")
    for (r, h), want in ref.items():
        assert np.allclose(out[r, h * 256:(h + 1) * 256], want, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- R1 = flash with integer max
def _flash_integer_max(q_hat, k_hat, v, vis, tile):
    """A flash pass in the kernels' recurrence: running max snapped to an integer in
    log2 units, P = bf16(2^(t - M)), lazy power-of-two rescale of O and l."""
    n, T = vis.shape
    out = np.zeros((n, v.shape[1]))
    for i in range(n):
        M, l, o = None, 0.0, np.zeros(v.shape[1])
        for j0 in range(0, T, tile):
            idx = [j for j in range(j0, min(T, j0 + tile)) if vis[i, j]]
            if not idx:
                continue
            t = np.array([O.bf16(q_hat[i] @ k_hat[j]) / 16.0 * math.log2(math.e) for j in idx])
            need = math.ceil(t.max())
            if M is None:
                M = need
            elif need > M + 8:
                o *= 2.0 ** (M - need)
                l *= 2.0 ** (M - need)
                M = need
            p = O.bf16(2.0 ** (t - M))
            l += p.sum()
            o += p @ v[idx]
        out[i] = o / l
    return O.bf16(out)


def test_r1_is_flash_with_integer_max_any_tile():
    rng = np.random.default_rng(7)
    n, T = 5, 40
    q = O.bf16(3 * rng.standard_normal((n, 256)))
    k = O.bf16(rng.standard_normal((T, 256)))
    v = O.bf16(rng.standard_normal((T, 256)))
    vis = O.visibility("causal", np.arange(n) + 30, T)
    g = np.full((n, 256), 30.0)                       # sigmoid rounds to exactly 1.0
    want, _, _ = O.attend_head(q, g, k, v, vis)
    for tile in (3, 8, 16):
        got = _flash_integer_max(q, k, v, vis, tile)
        assert np.allclose(got, want, rtol=0, atol=0) or \
            np.all(O.within_tolerance(got, want, 1.0, 0.0))


# ---------------------------------------------------------------- closed forms and invariants
def _prepared(S=16, seed=21, T=None):
    T = T or S
    qg, k, v, w_q, w_k = synth.attention_inputs(seed, S, T)
    f = lambda t: t.double().numpy()
    qg, k, v, w_q, w_k = f(qg), f(k), f(v), f(w_q), f(w_k)
    c, s = O.rope_tables(max(S, T))
    return qg, O.prep_keys(k, w_k, c, s), v, w_q, c, s


def test_zero_query_gives_mean_of_visible_values():
    qg, kp, v, w_q, c, s = _prepared()
    qg[:, :, :256] = 0.0                          # q = 0: every score is 0, every w_hat 1
    out = O.prefill(qg, kp, v, w_q, c, s, 0, 16)
    for r in [0, 5, 15]:
        for h in [0, 13]:
            kv = h // 12
            o = O.bf16(v[: r + 1, kv].mean(axis=0))
            want = O.bf16(o * O.bf16(1 / (1 + np.exp(-qg[r, h, 256:]))))
            assert np.array_equal(out[r, h * 256:(h + 1) * 256], want)


def test_constant_values_pass_through():
    qg, kp, v, w_q, c, s = _prepared()
    v[:, 0] = v[3, 0]
    v[:, 1] = v[7, 1]
    qg[:, :, 256:] = 30.0                          # sigmoid(30) rounds to 1.0
    out = O.prefill(qg, kp, v, w_q, c, s, 0, 16)
    for h in range(24):
        assert np.all(out[:, h * 256:(h + 1) * 256] == v[3 if h < 12 else 7, h // 12])


def test_single_visible_key_outputs_gated_value():
    """The first causal row sees only key 0: out = bf16(v_0 * bf16(sigmoid(g)))."""
    qg, kp, v, w_q, c, s = _prepared()
    out = O.prefill(qg, kp, v, w_q, c, s, 0, 16)
    for h in range(24):
        g = qg[0, h, 256:]
        want = O.bf16(v[0, h // 12] * O.bf16(1 / (1 + np.exp(-g))))
        assert np.array_equal(out[0, h * 256:(h + 1) * 256], want)


def test_gate_zero_halves_saturated_gate():
    qg, kp, v, w_q, c, s = _prepared()
    qg[:, :, 256:] = 0.0
    half = O.prefill(qg, kp, v, w_q, c, s, 0, 16)
    qg[:, :, 256:] = 30.0
    full = O.prefill(qg, kp, v, w_q, c, s, 0, 16)
    assert np.array_equal(half, full / 2)


def test_future_and_masked_keys_do_not_matter():
    qg, kp, v, w_q, c, s = _prepared()
    base = O.prefill(qg, kp, v, w_q, c, s, 0, 16)
    kp2, v2 = kp.copy(), v.copy()
    kp2[10:] += 3.0
    v2[10:] = -v2[10:]
    pert = O.prefill(qg, kp2, v2, w_q, c, s, 0, 16)
    assert np.array_equal(base[:10], pert[:10]) and not np.array_equal(base[10:], pert[10:])
    mask = (np.random.default_rng(8).random((16, 16)) < 0.4).astype(np.uint8)
    mask[np.arange(16), np.arange(16)] = 1
    m1, _, _ = O.masked(qg, kp, v, w_q, c, s, 0, 16, mask)
    kp3, v3 = kp.copy(), v.copy()
    hid = np.nonzero(mask[5] == 0)[0]
    kp3[hid] += 5.0
    v3[hid] *= 3.0
    m2, _, _ = O.masked(qg, kp3, v3, w_q, c, s, 0, 16, mask)
    assert np.array_equal(m1[5], m2[5])


def test_windows_equal_full_pass_rows():
    """[WIDE] §Test Plan: prefix windows at q_base 64/128/1,024 match the full pass."""
    S = 1088
    qg, kp, v, w_q, c, s = _prepared(S=S, seed=22)
    rows = np.array([0, 1, 63, 64, 127, 128, 500, 1023, 1024, 1087])
    full = O.prefill(qg, kp, v, w_q, c, s, 0, S, rows=rows, heads=[0, 23])
    for qb in (64, 128, 1024):
        sel = rows[rows >= qb]
        win = O.prefill(qg[qb:], kp, v, w_q, c, s, qb, S, rows=sel - qb, heads=[0, 23])
        assert np.array_equal(win, full[rows >= qb])


def test_bidirectional_and_causal_equal_masked():
    qg, kp, v, w_q, c, s = _prepared()
    bi = O.prefill(qg, kp, v, w_q, c, s, 0, 16, causal=False)
    mb, _, _ = O.masked(qg, kp, v, w_q, c, s, 0, 16, np.ones((16, 16), np.uint8))
    assert np.array_equal(bi, mb)
    ca = O.prefill(qg, kp, v, w_q, c, s, 0, 16)
    mc, _, _ = O.masked(qg, kp, v, w_q, c, s, 0, 16, np.tril(np.ones((16, 16), np.uint8)))
    assert np.array_equal(ca, mc)


def test_weights_rows_sum_to_one_and_hidden_are_zero():
    """[QSA] review F2: each head's weights sum to 1 within 2e-3; blocked positions carry
    exactly zero mass (the dump script's zero-mass assertion)."""
    qg, kp, v, w_q, c, s = _prepared(S=64, seed=23)
    mask = (np.random.default_rng(9).random((64, 64)) < 0.3).astype(np.uint8)
    mask[np.arange(64), np.arange(64)] = 1
    mask[7] = 0                                     # a fully hidden row
    out, w, hid = O.masked(qg, kp, v, w_q, c, s, 0, 64, mask, want_weights=True)
    assert hid[7] and hid.sum() == 1 and np.all(out[7] == 0) and np.all(w[:, 7] == 0)
    vis = mask != 0
    assert np.all(w[:, ~vis] == 0)
    # each weight is bf16(w_hat / L) and sum_j w_hat_j / L = 1, so a row misses 1 by at
    # most half an ulp per visible weight
    sums = w.sum(axis=2)[:, ~hid]
    bound = 0.5 * np.where(vis[None], O.ulp_bf16(w), 0.0).sum(axis=2)[:, ~hid]
    assert np.all(np.abs(sums - 1) <= bound + 1e-12)


def test_token_cap_row_weights_sum_to_one():
    """[QSA] review F2: one query row over exactly 8192 all-visible keys; every head's
    8192 weights are finite and sum to 1 within 2e-3."""
    S = 8192
    qg, k, v, w_q, w_k = synth.attention_inputs(25, 1, S)
    f = lambda t: t.double().numpy()
    qg, k, v, w_q, w_k = f(qg), f(k), f(v), f(w_q), f(w_k)
    c, s = O.rope_tables(S)
    kp = O.prep_keys(k, w_k, c, s)
    out, w, hid = O.masked(qg, kp, v, w_q, c, s, S - 1, S, np.ones((1, S), np.uint8),
                           want_weights=True)
    assert np.all(np.isfinite(w)) and not hid.any()
    assert np.all(np.abs(w.sum(axis=2) - 1) <= 2e-3)


def test_verify_equals_prefill_rows():
    L, R = 40, 4
    qg_all, kp, v, w_q, c, s = _prepared(S=L + R, seed=24)
    qg = qg_all[L:][None]
    out = O.verify(qg, kp[None], v[None], [L], w_q, c, s)
    full = O.prefill(qg_all, kp, v, w_q, c, s, 0, L + R)
    assert np.array_equal(out[0], full[L:])


def test_gather_pages_indexing():
    """Every gathered row carries its own (page, slot) label: position t comes from page
    table[t // page_size], slot t % page_size, for page sizes of one and two tiles."""
    rng = np.random.default_rng(5)
    for page_size in (128, 256):
        n_pages = 7
        pool = np.zeros((n_pages, page_size, 2))
        pool[:, :, 0] = np.arange(n_pages)[:, None]
        pool[:, :, 1] = np.arange(page_size)[None, :]
        table = rng.permutation(n_pages)
        n_tok = 3 * page_size + 37
        got = O.gather_pages(pool, table, n_tok, page_size)
        t = np.arange(n_tok)
        assert np.array_equal(got[:, 0], table[t // page_size])
        assert np.array_equal(got[:, 1], t % page_size)
    assert O.gather_pages(pool, table, 0, 256).shape == (0, 2)


def test_verify_paged_equals_contiguous_and_decode_equals_prefill_row():
    """Scattered pages give the contiguous cache's outputs bit for bit, and a one-row
    decode at position L equals row L of the full causal pass."""
    L, R, page_size = 300, 3, 128
    qg_all, kp, v, w_q, c, s = _prepared(S=L + R, seed=27)
    n_pages = 5
    order = np.array([3, 0, 4, 1, 2])                 # page order[i] holds positions i*128..
    kpool = np.zeros((n_pages, page_size, 2, 256))
    vpool = np.zeros_like(kpool)
    for i in range(-(-(L + R) // page_size)):
        rows = slice(i * page_size, min((i + 1) * page_size, L + R))
        n = rows.stop - rows.start
        kpool[order[i], :n] = kp[rows]
        vpool[order[i], :n] = v[rows]
    qg = qg_all[L:][None]
    paged = O.verify_paged(qg, kpool, vpool, order[None], page_size, [L], w_q, c, s)
    cont = O.verify(qg, kp[None], v[None], [L], w_q, c, s)
    assert np.array_equal(paged, cont)
    dec = O.verify_paged(qg_all[L:L + 1][None], kpool, vpool, order[None], page_size, [L],
                         w_q, c, s)
    full = O.prefill(qg_all, kp, v, w_q, c, s, 0, L + R)
    assert np.array_equal(dec[0, 0], full[L])


def _e4m3_grid():
    """Every finite OCP FP8 E4M3 value, decoded from its byte by the format's definition."""
    vals = []
    for byte in range(256):
        sign = -1.0 if byte >> 7 else 1.0
        e, m = (byte >> 3) & 15, byte & 7
        if e == 15 and m == 7:
            continue                                  # the NaN codes
        vals.append(sign * (m / 8) * 2.0 ** -6 if e == 0 else sign * (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(sorted(set(vals)))


def test_e4m3_grid_nearest_ties_to_even_and_saturation():
    """e4m3() keeps every grid value, returns the nearest grid value for random inputs (ties
    to the even mantissa, found by exhaustive search), and saturates at +-448."""
    grid = _e4m3_grid()
    assert grid.size == 253 and grid.max() == 448.0 and np.min(grid[grid > 0]) == 2.0 ** -9
    assert np.array_equal(O.e4m3(grid), grid)
    rng = np.random.default_rng(8)
    v = np.concatenate([rng.normal(size=4000) * 2.0 ** rng.integers(-12, 9, 4000),
                        (grid[1:] + grid[:-1]) / 2])  # includes every midpoint
    v = v[np.abs(v) <= 448]
    got = O.e4m3(v)
    d = np.abs(v[:, None] - grid[None, :])
    best = d.min(axis=1)
    for i in range(v.size):
        cand = grid[np.isclose(d[i], best[i], rtol=0, atol=0)]
        if cand.size == 1:
            assert got[i] == cand[0], v[i]
        else:                                         # a tie: the even mantissa (code) wins
            codes = [int(np.round(abs(c) / 2.0 ** (max(np.floor(np.log2(abs(c))), -6) - 3))) % 2
                     if c != 0 else 0 for c in cand]
            assert got[i] == cand[codes.index(0)], v[i]
    assert O.e4m3(463.99) == 448 and O.e4m3(464.0) == 448 and O.e4m3(1e9) == 448
    assert O.e4m3(-1e9) == -448 and O.e4m3(0.0) == 0


def test_e4m3_rows_scale_and_round_trip():
    """A row whose largest magnitude is 448 has scale 1, so its codes are e4m3 of the row
    itself (1.0625 ties down to 1.0, 1.1875 up to 1.25); the largest element of any row
    maps to +-448; a zero row gives scale 0 and zeros; the widened row is within 2^-4
    relative (plus one bf16 rounding) of the row for elements above the subnormal range."""
    row = np.zeros(256)
    row[:5] = [448.0, 1.0625, 1.1875, -3.0, 0.5]
    q, sc = O.quantize_e4m3_rows(row[None])
    assert sc[0] == 1.0
    assert list(q[0, :5]) == [448.0, 1.0, 1.25, -3.0, 0.5]
    assert np.array_equal(O.dequantize_e4m3_rows(q, sc)[0, :5], [448.0, 1.0, 1.25, -3.0, 0.5])
    rng = np.random.default_rng(9)
    x = O.bf16(rng.normal(size=(64, 256)) * 2.0 ** rng.integers(-8, 8, (64, 1)))
    q, sc = O.quantize_e4m3_rows(x)
    assert np.all(np.abs(q).max(axis=1) == 448.0)
    assert np.all(sc == O.fp32(np.abs(x).max(axis=1) / 448.0))
    xh = O.dequantize_e4m3_rows(q, sc)
    big = np.abs(x) >= 2.0 ** -6 * sc[:, None] * 1.0001
    rel = np.abs(xh - x)[big] / np.abs(x)[big]
    assert rel.max() <= 2.0 ** -4 * (1 + 2.0 ** -7) + 2.0 ** -8
    q0, sc0 = O.quantize_e4m3_rows(np.zeros((2, 256)))
    assert np.all(q0 == 0) and np.all(sc0 == 0) and np.all(O.dequantize_e4m3_rows(q0, sc0) == 0)


# ---------------------------------------------------------------- planted mistakes
def test_planted_unrounded_sigmoid_is_caught(monkeypatch):
    """[QSA] §Validation, mutation calibration: dropping the sigmoid's bf16 rounding
    must break an exact check."""
    monkeypatch.setattr(O, "sigmoid_gate", lambda g, mode="R1": 1.0 / (1.0 + np.exp(-g)))
    with pytest.raises(AssertionError):
        test_single_visible_key_outputs_gated_value()


def test_planted_kv_swap_is_caught(monkeypatch):
    """[QSA] §Validation: exchanging the two KV heads must fail."""
    monkeypatch.setattr(O, "GROUP", 1000)        # every head reads KV head 0
    with pytest.raises(AssertionError):
        test_f64_mode_equals_mp_bruteforce("causal", 0)


def test_planted_interleaved_rope_is_caught(monkeypatch):
    def interleaved(x, cos_rows, sin_rows, rounded=True):
        x = np.asarray(x, dtype=np.float64)
        y = x.copy()
        a, b = x[..., 0:64:2], x[..., 1:64:2]
        y[..., 0:64:2] = a * cos_rows - b * sin_rows
        y[..., 1:64:2] = b * cos_rows + a * sin_rows
        return y
    monkeypatch.setattr(O, "rope_partial", interleaved)
    with pytest.raises(AssertionError):
        test_rope_pairing_closed_form()


def test_planted_single_rounding_rope_is_caught(monkeypatch):
    """Rotating with one rounding of the exact a*c - b*s (and b*c + a*s) instead of
    rounding each product and then the sum must fail the hand-worked rounding pin."""
    def fused(x, cos_rows, sin_rows, rounded=True):
        x = np.asarray(x, dtype=np.float64)
        a, b = x[..., :32], x[..., 32:64]
        y = x.copy()
        y[..., :32] = a * cos_rows - b * sin_rows
        y[..., 32:64] = b * cos_rows + a * sin_rows
        return O.bf16(y) if rounded else y
    monkeypatch.setattr(O, "rope_partial", fused)
    with pytest.raises(AssertionError):
        test_rope_rounding_points_hand_worked()


def test_planted_unrounded_products_rope_is_caught(monkeypatch):
    """Rounding only the sum (products kept exact) must fail the same pin."""
    def sum_only(x, cos_rows, sin_rows, rounded=True):
        x = np.asarray(x, dtype=np.float64)
        a, b = x[..., :32], x[..., 32:64]
        y = x.copy()
        y[..., :32] = O.bf16(a * cos_rows - O.bf16(b * sin_rows))
        y[..., 32:64] = O.bf16(O.bf16(b * cos_rows) + a * sin_rows)
        return y
    monkeypatch.setattr(O, "rope_partial", sum_only)
    with pytest.raises(AssertionError):
        test_rope_rounding_points_hand_worked()


def test_planted_causal_for_sparse_mask_is_caught(monkeypatch):
    """[QSA] §Validation: replacing the stored mask with plain causality must fail."""
    real = O.visibility
    monkeypatch.setattr(O, "visibility",
                        lambda kind, rows, T, q_base=0, mask=None: real("causal", rows, T, q_base))
    with pytest.raises(AssertionError):
        test_masked_f64_equals_mp_bruteforce()


def test_planted_eps_outside_sqrt_is_caught(monkeypatch):
    def wrong(x, w, eps=O.EPS, rounded=True):
        x = np.asarray(x, dtype=np.float64)
        y = x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * (1.0 + w)
        return O.bf16(y) if rounded else y
    monkeypatch.setattr(O, "rms_norm_1pw", wrong)
    with pytest.raises(AssertionError):
        test_norm_constant_vector_closed_form()


# ---------------------------------------------------------------- selection mask
def _kept_blocks(mask_row, p):
    """Blocks kept in a mask row: every candidate block b has its first key 4b <= p."""
    nc = p // O.BLOCK_TOKENS + 1
    return {b for b in range(nc) if b * O.BLOCK_TOKENS < mask_row.shape[0]
            and mask_row[b * O.BLOCK_TOKENS]}


def test_select_brute_force_tiny():
    """Brute force over every subset: among the candidate subsets of size min(k, nc),
    exactly one is closed under 'beats' (higher score, or equal score and lower index)
    against every left-out candidate, and it is the oracle's. Scores are drawn from a
    handful of values (with -0, +0 and +-inf) so ties are everywhere."""
    import itertools
    rng = np.random.default_rng(81)
    vals = np.array([-np.inf, -1.0, -0.0, 0.0, 0.5, 1.0, np.inf])
    for trial in range(60):
        T = int(rng.integers(1, 27))
        nb = -(-T // O.BLOCK_TOKENS)
        q_base = int(rng.integers(0, T))
        rows = T - q_base
        k = int(rng.integers(1, 8))
        s = vals[rng.integers(0, len(vals), (rows, nb))]
        m = O.select_blocks_mask(s, q_base, T, k)
        for r in range(rows):
            p = q_base + r
            nc = min(nb, p // O.BLOCK_TOKENS + 1)
            beats = lambda a, b: s[r, a] > s[r, b] or (s[r, a] == s[r, b] and a < b)
            ok = [set(c) for c in itertools.combinations(range(nc), min(k, nc))
                  if all(beats(a, b) for a in c for b in set(range(nc)) - set(c))]
            assert len(ok) == 1, (trial, r)
            assert _kept_blocks(m[r], p) == ok[0], (trial, r)
            assert np.array_equal(m[r] != 0, (np.arange(T) <= p) &
                                  np.isin(np.arange(T) // O.BLOCK_TOKENS, list(ok[0])))


def test_select_invariants_and_special_cases():
    """N(0,1) scores, a ragged T: the mask lies inside causality, keeps min(k, nc) blocks,
    never hides a whole row; k >= nc gives the causal row; k = 1 keeps numpy's argmax
    (its first maximum, i.e. the lower index on a tie); constant scores keep the k lowest
    blocks; raising a kept block's score or lowering a dropped one changes nothing."""
    rng = np.random.default_rng(82)
    T, q_base, k = 1203, 5, 37
    rows = T - q_base
    nb = -(-T // 4)
    s = rng.standard_normal((rows, nb))
    m = O.select_blocks_mask(s, q_base, T, k)
    causal = O.visibility("causal", np.arange(rows), T, q_base)
    assert not np.any((m != 0) & ~causal)
    for r in range(0, rows, 7):
        p = q_base + r
        nc = min(nb, p // 4 + 1)
        kept = _kept_blocks(m[r], p)
        assert len(kept) == min(k, nc) and m[r].any()
        if k >= nc:
            assert np.array_equal(m[r] != 0, causal[r])
        else:
            lowest_kept = min(s[r, b] for b in kept)
            assert all(s[r, b] <= lowest_kept for b in set(range(nc)) - kept)
    one = O.select_blocks_mask(s, q_base, T, 1)
    for r in range(0, rows, 11):
        p = q_base + r
        assert _kept_blocks(one[r], p) == {int(np.argmax(s[r, :min(nb, p // 4 + 1)]))}
    const = O.select_blocks_mask(np.full((rows, nb), 0.25), q_base, T, k)
    j = np.arange(T)
    assert np.array_equal(const != 0, causal & (j < 4 * k)[None, :])
    assert np.array_equal(O.select_blocks_mask(s, q_base, T, nb) != 0, causal)
    s2 = s.copy()
    r = rows - 1
    kept = sorted(_kept_blocks(m[r], q_base + r))
    dropped = sorted(set(range(nb)) - set(kept))
    s2[r, kept[0]] += 5.0
    s2[r, dropped[0]] -= 5.0
    assert np.array_equal(O.select_blocks_mask(s2[r:], q_base + r, T, k), m[r:])


def test_planted_reversed_tie_rule_is_caught():
    """An oracle that breaks ties toward the higher block index fails the constant-score
    special case (the k lowest blocks)."""
    T, k = 40, 3
    s = np.zeros((1, 10))
    m = O.select_blocks_mask(s, T - 1, T, k)
    order_hi = np.lexsort((-np.arange(10), -s[0]))[:k]      # the planted rule
    planted = np.isin(np.arange(T) // 4, order_hi)
    assert not np.array_equal(m[0] != 0, planted)
    assert np.array_equal(m[0] != 0, np.arange(T) < 4 * k)


def test_select_window_rows_equal_full_pass():
    """A row's selection depends only on its own scores and position: the rows of a window
    at q_base equal the same positions' rows of the full pass."""
    rng = np.random.default_rng(83)
    T, k = 700, 20
    s = rng.standard_normal((T, -(-T // 4)))
    full = O.select_blocks_mask(s, 0, T, k)
    for q_base, rows in ((0, 1), (64, 100), (333, 367), (699, 1)):
        win = O.select_blocks_mask(s[q_base:q_base + rows], q_base, T, k)
        assert np.array_equal(win, full[q_base:q_base + rows]), q_base
