"""Pins of the oracle's FP8 leg (e4m3 codes, per-row scales, FP8 indexer score).

The encodings below are worked out by hand from the OCP E4M3 definition
(bias 7, 3 mantissa bits, no infinities, largest finite 448); the reading
adds round-to-nearest with ties to the even code and saturation at +-448.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

# (value, code): normals, subnormals, the largest finite, signs, ties, saturation
HAND = [
    (1.0, 0x38),            # 0 0111 000
    (448.0, 0x7E),          # 1.75 * 2^8
    (2.0 ** -6, 0x08),      # smallest normal
    (2.0 ** -9, 0x01),      # smallest subnormal
    (7 * 2.0 ** -9, 0x07),  # largest subnormal
    (-2.0, 0xC0),
    (1.0625, 0x38),         # halfway 1.0 / 1.125 -> even mantissa 0
    (1.1875, 0x3A),         # halfway 1.125 / 1.25 -> even mantissa 2
    (3 * 2.0 ** -10, 0x02),  # halfway 2^-9 / 2^-8 -> even code
    (2.0 ** -11, 0x00),     # below half the smallest subnormal
    (500.0, 0x7E),          # saturates
    (-1e9, 0xFE),
    (0.0, 0x00),
    (-0.0, 0x80),
]


@pytest.mark.parametrize("x,code", HAND)
def test_e4m3_hand_encodings(x, code):
    assert oracle.e4m3_from_double(x) == code


def test_e4m3_values_round_trip_and_increase():
    vals = [oracle.e4m3_value(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))
    assert vals[-1] == 448.0 and np.isnan(oracle.e4m3_value(0x7F))
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.e4m3_from_double(oracle.e4m3_value(c)) == c


def test_e4m3_matches_an_independent_conversion_in_range():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(-448, 448, 3000), rng.normal(0, 1e-2, 3000),
                        rng.normal(0, 1.0, 3000)])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_double(v) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def test_quantize_rows_bounds():
    rng = np.random.default_rng(6)
    x = synth.bf16_bits(rng.normal(0, 3, (64, 64)).astype(np.float32))
    x[3] = 0  # an all-zero row
    code, scale = oracle.quantize_rows_e4m3(x)
    xv = synth.bf16_to_f32(x).astype(np.float64)
    assert scale[3] == 0 and not code[3].any()
    amax = np.abs(xv).max(axis=1)
    nz = amax > 0
    assert np.allclose(scale[nz], (amax[nz] / 448).astype(np.float32), rtol=0, atol=0)
    deq = np.vectorize(oracle.e4m3_value)(code).astype(np.float64) * scale[:, None]
    # within half an e4m3 step: 2^-4 relative for normals, 2^-10 * scale absolute below
    assert (np.abs(deq - xv) <= 2.0 ** -4 * np.abs(xv) + 2.0 ** -10 * scale[:, None]).all()
    # the row maximum lands on +-448 exactly
    arg = np.abs(xv).argmax(axis=1)
    assert (np.abs(deq[nz, arg[nz]]) == 448.0 * scale[nz].astype(np.float64)).all()


def _exact_case(rng, B, T, H_i, G, d=64):
    """Rows of e4m3-representable values whose maximum is 448 (scale exactly 1)."""
    def rows(n):
        c = rng.integers(0, 0x7E, (n, d)).astype(np.uint8) | rng.integers(0, 2, (n, d)).astype(
            np.uint8) << 7
        c[np.arange(n), rng.integers(0, d, n)] = 0x7E
        v = np.vectorize(oracle.e4m3_value)(c).astype(np.float32)
        return synth.bf16_bits(v)
    q = rows(B * T * H_i).reshape(B, T, H_i, d)
    k = rows(B * G).reshape(B, G, d)
    return q, k


def test_fp8_score_with_unit_scales_equals_the_bf16_score():
    rng = np.random.default_rng(7)
    B, T, H_i, G, P = 2, 3, 4, 40, 4
    q, k = _exact_case(rng, B, T, H_i, G)
    w = rng.uniform(0, 1, (B, T, H_i)).astype(np.float32)
    seq = np.array([G * P, (G - 7) * P], np.int32)
    cq, sq = oracle.quantize_rows_e4m3(q)
    ck, sk = oracle.quantize_rows_e4m3(k)
    assert (sq == 1).all() and (sk == 1).all()
    got = oracle.index_scores_e4m3(cq, sq, w, ck, sk, seq, P)
    ref = oracle.index_scores(q, w, k, seq, P)
    assert np.array_equal(got, ref)


def test_fp8_score_follows_the_key_scale():
    rng = np.random.default_rng(8)
    B, T, H_i, G, P = 1, 2, 4, 16, 4
    q, k = _exact_case(rng, B, T, H_i, G)
    w = rng.uniform(0, 1, (B, T, H_i)).astype(np.float32)
    seq = np.array([G * P], np.int32)
    cq, sq = oracle.quantize_rows_e4m3(q)
    ck, sk = oracle.quantize_rows_e4m3(k)
    base = oracle.index_scores_e4m3(cq, sq, w, ck, sk, seq, P)
    k2 = synth.bf16_bits(synth.bf16_to_f32(k) * np.float32(1.0 / 64))  # exact power of two
    ck2, sk2 = oracle.quantize_rows_e4m3(k2)
    assert np.array_equal(ck2, ck) and np.array_equal(sk2, sk / 64)
    got = oracle.index_scores_e4m3(cq, sq, w, ck2, sk2, seq, P)
    assert np.array_equal(got, (base.astype(np.float64) / 64).astype(np.float32))


# ---------------------------------------------------------------------------
# attention over an FP8 K/V cache (element = e4m3(code) * row scale)
# ---------------------------------------------------------------------------

def _kv8_case(seed, B=2, L=96, H_q=4, d_qk=16, d_v=8, k=10, P=4, pow2_scales=True):
    rng = np.random.default_rng(seed)
    kc = rng.integers(0, 0x7F, (B, L, d_qk)).astype(np.uint8) | (
        rng.integers(0, 2, (B, L, d_qk)).astype(np.uint8) << 7)
    vc = rng.integers(0, 0x7F, (B, L, d_v)).astype(np.uint8) | (
        rng.integers(0, 2, (B, L, d_v)).astype(np.uint8) << 7)
    if pow2_scales:
        ks = (2.0 ** rng.integers(-12, -6, (B, L))).astype(np.float32)
        vs = (2.0 ** rng.integers(-10, -4, (B, L))).astype(np.float32)
    else:
        ks = rng.uniform(0.001, 0.02, (B, L)).astype(np.float32)
        vs = rng.uniform(0.001, 0.02, (B, L)).astype(np.float32)
    q = synth.bf16_bits(rng.standard_normal((B, 1, H_q, d_qk)).astype(np.float32))
    seq = np.array([L, L - 13], np.int32)[:B]
    idx = np.full((B, 1, k), -1, np.int32)
    for b in range(B):
        G = int(seq[b]) // P
        idx[b, 0, :k - 2] = np.sort(rng.choice(G, k - 2, replace=False))
    return q, kc, ks, vc, vs, seq, idx


def _decode(codes, scales):
    vals = np.array([oracle.e4m3_value(c) for c in range(256)])
    return vals[codes] * scales[..., None].astype(np.float64)


def test_kv8_power_of_two_scales_equal_the_bf16_oracle():
    """With power-of-two scales every dequantized element is a bf16 value, so
    the FP8 attention must equal the bf16 oracle's bit for bit."""
    q, kc, ks, vc, vs, seq, idx = _kv8_case(400)
    Kf, Vf = _decode(kc, ks), _decode(vc, vs)
    Kb, Vb = synth.bf16_bits(Kf.astype(np.float32)), synth.bf16_bits(Vf.astype(np.float32))
    assert np.array_equal(synth.bf16_to_f32(Kb).astype(np.float64), Kf)
    assert np.array_equal(synth.bf16_to_f32(Vb).astype(np.float64), Vf)
    o8, l8 = oracle.sparse_attn_e4m3kv(q, kc, ks, vc, vs, seq, idx, 4, 0.25)
    ob, lb = oracle.sparse_attn(q, Kb, Vb, seq, idx, 4, 0.25)
    assert np.array_equal(o8, ob)
    assert np.array_equal(l8, lb)


def test_kv8_brute_force_softmax():
    """Arbitrary scales: a numpy softmax (scipy logsumexp) over the decoded
    rows of the selected tokens, rounded to bf16 the same way."""
    from scipy.special import logsumexp
    q, kc, ks, vc, vs, seq, idx = _kv8_case(401, pow2_scales=False)
    o8, l8 = oracle.sparse_attn_e4m3kv(q, kc, ks, vc, vs, seq, idx, 4, 0.3)
    Kf, Vf = _decode(kc, ks), _decode(vc, vs)
    qf = synth.bf16_to_f32(q).astype(np.float64)
    for b in range(q.shape[0]):
        G = int(seq[b]) // 4
        toks = [4 * g + i for g in idx[b, 0] if 0 <= g < G for i in range(4)]
        z = 0.3 * qf[b, 0] @ Kf[b, toks].T                      # [H_q][n]
        lse = logsumexp(z, axis=1)
        out = np.exp(z - lse[:, None]) @ Vf[b, toks]
        np.testing.assert_allclose(l8[b, 0], lse, rtol=1e-6)
        ref_bits = np.array([[oracle.bf16_from_double(x) for x in row] for row in out])
        assert np.array_equal(o8[b, 0], ref_bits)


def test_kv8_scales_belong_to_their_own_cache():
    """Swapping the key and value scales changes the result (each cache's
    scale multiplies its own elements only)."""
    q, kc, ks, vc, vs, seq, idx = _kv8_case(402)
    o1, _ = oracle.sparse_attn_e4m3kv(q, kc, ks, vc, vs, seq, idx, 4, 0.25)
    o2, _ = oracle.sparse_attn_e4m3kv(q, kc, vs, vc, ks, seq, idx, 4, 0.25)
    assert not np.array_equal(o1, o2)


# ------------------------------------------------------------- INT8 K/V ---
# Reading: symmetric codes in [-127, 127], one fp32 scale per row = amax / 127,
# code = nearest integer to x / scale with ties to the even integer.

def _i8_exact(x, scale):
    """The nearest integer to x / scale from exact rationals (ties to even)."""
    from fractions import Fraction
    r = Fraction(x) / Fraction(scale)
    n = int(r)  # toward zero
    if r < 0:
        n, frac = -int(-r), -r - int(-r)
    else:
        frac = r - n
    if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and abs(n) % 2 == 1):
        n += 1 if r >= 0 else -1
    return max(-127, min(127, n))


def test_i8_hand_encodings_at_unit_scale():
    """scale 1 (amax 127): codes are the rounded values themselves."""
    cases = [(2.5, 2), (3.5, 4), (-2.5, -2), (-3.5, -4), (0.5, 0), (1.5, 2), (126.5, 126),
             (127.0, 127), (-127.0, -127), (0.0, 0), (-0.25, 0), (7.75, 8)]
    for x, c in cases:
        assert oracle.i8_from_double(x, 1.0) == c, (x, c)


def test_i8_quantizer_matches_exact_rationals():
    rng = np.random.default_rng(410)
    x = synth.bf16_bits((rng.standard_normal((40, 24)) * 10.0 ** rng.integers(-3, 3, (40, 1)))
                        .astype(np.float32))
    code, scale = oracle.quantize_rows_i8(x)
    xf = synth.bf16_to_f32(x).astype(np.float64)
    from fractions import Fraction
    for r in range(x.shape[0]):
        amax = Fraction(float(np.abs(xf[r]).max())) / 127
        # the fp32 nearest to amax / 127: one of the two fp32 values around the double
        d = float(amax)
        cands = [np.float32(d), np.nextafter(np.float32(d), np.float32(np.inf)),
                 np.nextafter(np.float32(d), np.float32(-np.inf))]
        best = min(cands, key=lambda c: abs(Fraction(float(c)) - amax))
        assert scale[r] == best
        for i in range(x.shape[1]):
            assert code[r, i] == _i8_exact(float(xf[r, i]), float(scale[r])), (r, i)


def test_i8_rows_bounds():
    x = synth.bf16_bits(np.array([[0.0] * 8, [3.0, -6.0, 1.0, 0.0, 5.0, -1.0, 2.0, 6.0]],
                                 np.float32))
    code, scale = oracle.quantize_rows_i8(x)
    assert scale[0] == 0.0 and (code[0] == 0).all()  # zero row
    assert abs(int(code[1, 1])) == 127 and abs(int(code[1, 7])) == 127  # the amax elements
    assert code[1, 1] == -127 and code[1, 7] == 127
    assert np.float32(scale[1]) == np.float32(6.0 / 127.0)


def _i8_case(seed, B=2, L=96, H_q=4, d_qk=16, d_v=8, k=10, P=4):
    rng = np.random.default_rng(seed)
    kc = rng.integers(-127, 128, (B, L, d_qk)).astype(np.int8)
    vc = rng.integers(-127, 128, (B, L, d_v)).astype(np.int8)
    ks = rng.uniform(0.001, 0.02, (B, L)).astype(np.float32)
    vs = rng.uniform(0.001, 0.02, (B, L)).astype(np.float32)
    q = synth.bf16_bits(rng.standard_normal((B, 1, H_q, d_qk)).astype(np.float32))
    seq = np.array([L, L - 13], np.int32)[:B]
    idx = np.full((B, 1, k), -1, np.int32)
    for b in range(B):
        G = int(seq[b]) // P
        idx[b, 0, :k - 2] = np.sort(rng.choice(G, k - 2, replace=False))
        idx[b, 0, k - 2] = G + 1  # past the sequence: skipped
    return q, kc, ks, vc, vs, seq, idx


def test_i8kv_unit_scales_equal_the_bf16_oracle():
    """Scales 1 and codes that bf16 holds exactly (|c| <= 127 < 256): the INT8
    attention must equal the bf16 oracle on the integer-valued caches."""
    q, kc, ks, vc, vs, seq, idx = _i8_case(420)
    one_k, one_v = np.ones_like(ks), np.ones_like(vs)
    o8, l8 = oracle.sparse_attn_i8kv(q, kc, one_k, vc, one_v, seq, idx, 4, 0.01)
    Kb = synth.bf16_bits(kc.astype(np.float32))
    Vb = synth.bf16_bits(vc.astype(np.float32))
    ob, lb = oracle.sparse_attn(q, Kb, Vb, seq, idx, 4, 0.01)
    assert np.array_equal(o8, ob)
    assert np.array_equal(l8, lb)


def test_i8kv_brute_force_softmax():
    from scipy.special import logsumexp
    q, kc, ks, vc, vs, seq, idx = _i8_case(421)
    o8, l8 = oracle.sparse_attn_i8kv(q, kc, ks, vc, vs, seq, idx, 4, 0.3)
    Kf = kc.astype(np.float64) * ks[..., None].astype(np.float64)
    Vf = vc.astype(np.float64) * vs[..., None].astype(np.float64)
    qf = synth.bf16_to_f32(q).astype(np.float64)
    for b in range(q.shape[0]):
        G = int(seq[b]) // 4
        toks = [4 * g + i for g in idx[b, 0] if 0 <= g < G for i in range(4)]
        z = 0.3 * qf[b, 0] @ Kf[b, toks].T
        lse = logsumexp(z, axis=1)
        out = np.exp(z - lse[:, None]) @ Vf[b, toks]
        np.testing.assert_allclose(l8[b, 0], lse, rtol=1e-6)
        ref_bits = np.array([[oracle.bf16_from_double(x) for x in row] for row in out])
        assert np.array_equal(o8[b, 0], ref_bits)


def test_i8kv_power_of_two_rescaling():
    """Doubling every value scale doubles the output exactly; doubling every
    key scale while halving the softmax scale leaves the result unchanged."""
    q, kc, ks, vc, vs, seq, idx = _i8_case(422)
    o1, l1 = oracle.sparse_attn_i8kv(q, kc, ks, vc, vs, seq, idx, 4, 0.25)
    o2, l2 = oracle.sparse_attn_i8kv(q, kc, ks, vc, vs * 2, seq, idx, 4, 0.25)
    assert np.array_equal(synth.bf16_to_f32(o2), 2 * synth.bf16_to_f32(o1))
    assert np.array_equal(l1, l2)
    o3, l3 = oracle.sparse_attn_i8kv(q, kc, ks * 2, vc, vs, seq, idx, 4, 0.125)
    assert np.array_equal(o3, o1) and np.array_equal(l3, l1)
    o4, _ = oracle.sparse_attn_i8kv(q, kc, vs, vc, ks, seq, idx, 4, 0.25)
    assert not np.array_equal(o4, o1)
