"""Pins of the CPU oracle against things other than itself.

Each check ties an oracle function to a hand-derived worked example, an exact
rational computation, a closed form, a special case that reduces to a library
routine, or a brute-force enumeration, so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
import synth
from conftest import read_fixture

bf = synth.bf16_bits
unbf = synth.bf16_to_f32


def _bf_exact(x):
    """bf16 bits of a value that is exactly representable (checked)."""
    b = bf(np.array(x, np.float32))
    assert (unbf(b) == np.array(x, np.float32)).all()
    return b


def _bf16_neighbours(b):
    """The bf16 values just below and above the bf16 value with bits b (finite)."""
    v = float(unbf(np.array([b], np.uint16))[0])
    up = (int(b) + 1) & 0xFFFF if v >= 0 else (int(b) - 1) & 0xFFFF
    dn = (int(b) - 1) & 0xFFFF if v > 0 else (int(b) + 1) & 0xFFFF
    if v == 0:
        dn = 0x8001
        up = 0x0001
    f = lambda x: Fraction(float(unbf(np.array([x], np.uint16))[0]))
    return f(dn), Fraction(v), f(up)


# ---------------------------------------------------------------- bf16 ---

def test_bf16_rounding_matches_library_for_float32_values():
    # torch's float32 -> bfloat16 conversion rounds to nearest even
    import torch
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(4000).astype(np.float32),
                        (rng.standard_normal(1000) * 1e-38).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, -2.5, 3.0e38], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(v)) for v in x], np.uint16)
    assert (got == ref).all()


def test_bf16_rounding_ties_and_no_double_rounding():
    # exact midpoints go to the even neighbour
    assert oracle.bf16_from_double(1 + 2 ** -8) == 0x3F80
    assert oracle.bf16_from_double(1 + 3 * 2 ** -8) == 0x3F82
    assert oracle.bf16_from_double(-(1 + 2 ** -8)) == 0xBF80
    # just above a midpoint, by less than a float32 ulp: must round up, which a
    # double -> float32 -> bf16 chain would get wrong
    assert oracle.bf16_from_double(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert oracle.bf16_from_double(1 + 2 ** -8 - 2 ** -40) == 0x3F80


# ---------------------------------------------------------------- pool ---

def test_pool_worked_example():
    fx = read_fixture("indexpool_worked.txt")
    P, d = int(fx["P"][0]), int(fx["d"][0])
    k = np.array([[float(v) for v in fx[f"k{j}"]] for j in range(P)], np.float32)
    alpha = np.array([float(v) for v in fx["alpha"]], np.float32)
    expect = np.array([float(v) for v in fx["expect"]], np.float32)
    got = oracle.pool_keys(_bf_exact(k)[None], alpha[None, None], np.array([P], np.int32), P)
    assert got.shape == (1, 1, d)
    assert (got[0, 0] == _bf_exact(expect)).all()


@pytest.mark.parametrize("j", [0, 1, 2, 3])
def test_pool_one_hot_is_strided_subsample(j):
    spec = synth.Spec(B=2, lengths=[64, 40], H_i=2, pool_mode=f"onehot:{j}", seed=11)
    c = synth.generate(spec, with_kv=False)
    got = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    for b, L in enumerate(spec.lengths):
        G = L // 4
        assert (got[b, :G] == c["k_idx"][b, j:4 * G:4]).all()


def test_pool_uniform_is_mean():
    # QSA-style r=4 average pooling is the uniform-weight special case
    spec = synth.Spec(B=1, lengths=[256], idx_values="int3", pool_mode="uniform", seed=12)
    c = synth.generate(spec, with_kv=False)
    got = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    kf = unbf(c["k_idx"][0]).reshape(64, 4, 64).astype(np.float64)
    mean = kf.mean(axis=1)  # multiples of 1/4, exact in bf16
    assert (unbf(got[0]).astype(np.float64) == mean).all()


def test_pool_dyadic_integer_keys_exact():
    # tiny-workload recipe: kbar = (4a + 2b + c + d) / 8 in integers
    spec = synth.named("tiny")
    spec = synth.Spec(**{**spec.__dict__, "lengths": [512]})
    c = synth.generate(spec, with_kv=False)
    got = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    ki = unbf(c["k_idx"][0]).astype(np.int64).reshape(128, 4, 64)
    num = 4 * ki[:, 0] + 2 * ki[:, 1] + ki[:, 2] + ki[:, 3]
    assert (unbf(got[0]).astype(np.float64) == num / 8.0).all()


def test_pool_gaussian_is_nearest_bf16_of_exact_sum():
    spec = synth.Spec(B=1, lengths=[64], pool_mode="softmax", seed=13)
    c = synth.generate(spec, with_kv=False)
    got = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    k = unbf(c["k_idx"][0])
    for g in range(16):
        for i in range(0, 64, 3):
            exact = sum(Fraction(float(c["pool_w"][0, g, j])) * Fraction(float(k[4 * g + j, i]))
                        for j in range(4))
            lo, mid, hi = _bf16_neighbours(got[0, g, i])
            assert abs(exact - mid) <= abs(exact - lo) and abs(exact - mid) <= abs(exact - hi)
            if abs(exact - mid) == abs(exact - lo) or abs(exact - mid) == abs(exact - hi):
                assert int(got[0, g, i]) % 2 == 0  # tie -> even mantissa


def test_pool_hard_sums_round_exactly():
    """Sums on or a hair beside a bf16 midpoint, after cancellation, or spanning
    hundreds of binades: the pooled key is the nearest bf16 of the exact
    rational sum (ties to even), with no double rounding."""
    import pool_cases
    cs = pool_cases.cases()
    k_idx, pool_w = pool_cases.as_arrays(cs, d=8)
    got = oracle.pool_keys(k_idx, pool_w, np.array([k_idx.shape[1]], np.int32), 4)
    for g, (a, k) in enumerate(cs):
        want = pool_cases.round_bf16(pool_cases.exact_sum(a, k))
        assert (got[0, g] == want).all(), (g, a, k, got[0, g, 0], want)


def test_pool_hand_worked_hard_sums():
    # worked by hand from the bf16 format (8 significant bits, ties to even):
    #   (1 + 2^-8) * 1 + 2^-60 * 1  lies just above the midpoint of 1 and
    #   1 + 2^-7, so it rounds up to 1 + 2^-7 = 0x3F81 (a sum formed in double
    #   would drop the 2^-60 and tie down to 1.0);
    #   1 * 1 + 2^-8 * 1 is exactly that midpoint: ties to even, 1.0 = 0x3F80;
    #   1 * (1 + 2^-7) + 2^-8 * 1 is the midpoint of 1 + 2^-7 and 1 + 2^-6:
    #   ties to the even mantissa, 1 + 2^-6 = 0x3F82;
    #   2^100 - 2^100 + 3 - 2^-130 lies just below 3 = 0x4040;
    #   -(1 + 2^-8) + -(2^-70) rounds away from zero to -(1 + 2^-7) = 0xBF81;
    #   -1 - 2^-8 is exactly a midpoint: ties to even, -1.0 = 0xBF80.
    one, rows = 0x3F80, []
    rows.append(([1 + 2 ** -8, 2 ** -60, 0, 0], [one, one, 0, 0], 0x3F81))
    rows.append(([1, 2 ** -8, 0, 0], [one, one, 0, 0], 0x3F80))
    rows.append(([1, 2 ** -8, 0, 0], [0x3F81, one, 0, 0], 0x3F82))
    rows.append(([1, 1, 1, 2 ** -130], [0x7180, 0xF180, 0x4040, 0xBF80], 0x4040))
    rows.append(([1 + 2 ** -8, 2 ** -70, 0, 0], [0xBF80, 0xBF80, 0, 0], 0xBF81))
    rows.append(([1, 2 ** -8, 0, 0], [0xBF80, 0xBF80, 0, 0], 0xBF80))
    for a, k, want in rows:
        got = oracle.pool_keys(np.array(k, np.uint16).reshape(1, 4, 1),
                               np.array(a, np.float32).reshape(1, 1, 4),
                               np.array([4], np.int32), 4)
        assert int(got[0, 0, 0]) == want, (a, k, hex(int(got[0, 0, 0])), hex(want))


def test_pool_p1_identity_and_tail_untouched():
    spec = synth.Spec(B=1, lengths=[30], P=1, pool_mode="dyadic", seed=14)
    c = synth.generate(spec, with_kv=False)
    got = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 1)
    assert (got[0, :30] == c["k_idx"][0, :30]).all()
    # P=4 with L=30: 7 complete groups; the partial tail group is not pooled
    spec4 = synth.Spec(B=1, lengths=[30], L_cap=32, P=4, pool_mode="softmax", seed=14)
    c4 = synth.generate(spec4, with_kv=False)
    out = np.full((1, 8, 64), 0x1234, np.uint16)
    oracle.pool_keys(c4["k_idx"], c4["pool_w"], c4["seq_len"], 4, out=out)
    assert (out[0, 7] == 0x1234).all() and (out[0, :7] != 0x1234).any()


# --------------------------------------------------------------- score ---

def test_score_worked_example():
    fx = read_fixture("indexer_topk_worked.txt")
    H, d = int(fx["H"][0]), int(fx["d"][0])
    q = np.array([[float(v) for v in fx[f"q{h}"]] for h in range(H)], np.float32)
    w = np.array([float(v) for v in fx["w"]], np.float32)
    kb = np.array([[float(v) for v in fx[f"kbar{g}"]] for g in range(4)], np.float32)
    s = oracle.index_scores(_bf_exact(q)[None, None], w[None, None], _bf_exact(kb)[None],
                            np.array([16], np.int32), 4)
    assert (s[0, 0] == np.array([float(v) for v in fx["scores"]], np.float32)).all()


def test_score_exact_rational_brute_force():
    spec = synth.Spec(B=2, lengths=[64, 48], T=2, H_i=3, w_mode="signed", seed=15)
    c = synth.generate(spec, with_kv=False)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    s = oracle.index_scores(c["q_idx"], c["w_head"], kp, c["seq_len"], 4)
    qf, kf = unbf(c["q_idx"]), unbf(kp)
    for b in range(2):
        G = spec.lengths[b] // 4
        for t in range(2):
            for g in range(kp.shape[1]):
                if g >= G:
                    assert s[b, t, g] == -np.inf
                    continue
                exact = Fraction(0)
                for h in range(3):
                    dot = sum(Fraction(float(qf[b, t, h, i])) * Fraction(float(kf[b, g, i]))
                              for i in range(64))
                    exact += Fraction(float(c["w_head"][b, t, h])) * max(dot, Fraction(0))
                got = Fraction(float(s[b, t, g]))
                ulp = Fraction(float(np.spacing(np.float32(abs(float(exact)) or 1e-30))))
                assert abs(got - exact) <= ulp / 2


def test_score_one_hot_head_weight_is_relu_dot():
    spec = synth.Spec(B=1, lengths=[400], H_i=8, w_mode="onehot:5", seed=16)
    c = synth.generate(spec, with_kv=False)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    s = oracle.index_scores(c["q_idx"], c["w_head"], kp, c["seq_len"], 4)
    dots = unbf(kp[0]).astype(np.float64) @ unbf(c["q_idx"][0, 0, 5]).astype(np.float64)
    assert np.array_equal(s[0, 0], np.maximum(dots, 0).astype(np.float32))


def test_score_p1_is_unpooled_indexer():
    spec = synth.Spec(B=1, lengths=[128], P=1, H_i=4, pool_mode="dyadic", seed=17)
    c = synth.generate(spec, with_kv=False)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 1)
    s_pool = oracle.index_scores(c["q_idx"], c["w_head"], kp, c["seq_len"], 1)
    s_raw = oracle.index_scores(c["q_idx"], c["w_head"], c["k_idx"], c["seq_len"], 1)
    assert np.array_equal(s_pool, s_raw)
    q = unbf(c["q_idx"][0, 0]).astype(np.float64)          # [H][d]
    k = unbf(c["k_idx"][0]).astype(np.float64)             # [L][d]
    ref = (np.maximum(k @ q.T, 0) * c["w_head"][0, 0].astype(np.float64)).sum(axis=1)
    assert np.allclose(s_raw[0, 0], ref, rtol=1e-6, atol=1e-6)


def test_score_causal_group_mask_and_positive_zero():
    spec = synth.Spec(B=1, lengths=[64], T=5, prefill=True, H_i=2, w_mode="signed", seed=18)
    c = synth.generate(spec, with_kv=False)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    s = oracle.index_scores(c["q_idx"], c["w_head"], kp, c["seq_len"], 4, q_pos=c["q_pos"])
    for t, p in enumerate(c["q_pos"][0]):
        n = (int(p) + 1) // 4   # groups whose last token 4g+3 <= p
        assert np.isfinite(s[0, t, :n]).all() and (s[0, t, n:] == -np.inf).all()
    # an all-negative dot product row: score is +0, never -0
    q = np.zeros((1, 1, 2, 64), np.float32); q[..., 0] = 1.0
    k = np.zeros((1, 4, 64), np.float32); k[0, :, 0] = -1.0
    w = np.array([[[-1.0, 2.0]]], np.float32)
    s0 = oracle.index_scores(_bf_exact(q), w, _bf_exact(k), np.array([16], np.int32), 4)
    assert (s0 == 0).all() and not np.signbit(s0).any()


# -------------------------------------------------------------- select ---

def _brute_topk(row, n, k):
    order = sorted(range(n), key=lambda g: (-float(row[g]), g))[:k]
    return sorted(order) + [-1] * (k - min(k, n))


def test_topk_worked_example():
    fx = read_fixture("indexer_topk_worked.txt")
    s = np.array([float(v) for v in fx["scores"]], np.float32)[None]
    for k in (2, 3, 4, 6):
        got = oracle.topk(s, np.array([4], np.int32), k)
        assert got[0].tolist() == [int(v) for v in fx[f"top{k}"]]
    ts = np.array([float(v) for v in fx["tie_scores"]], np.float32)[None]
    for k in (2, 4):
        got = oracle.topk(ts, np.array([5], np.int32), k)
        assert got[0].tolist() == [int(v) for v in fx[f"tie_top{k}"]]


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(19)
    for trial in range(60):
        G = int(rng.integers(1, 300))
        n = int(rng.integers(0, G + 1))
        k = int(rng.integers(1, 80))
        row = rng.integers(-4, 5, size=G).astype(np.float32)       # many ties
        if trial % 3 == 0:
            row = (rng.standard_normal(G) * 3).astype(np.float32)
        row[rng.random(G) < 0.1] = -0.0
        got = oracle.topk(row[None], np.array([n], np.int32), k)
        assert got[0].tolist() == _brute_topk(row, n, k)


def test_topk_all_when_k_covers_valid():
    row = np.array([3, 1, 2, 5, 4, 0, 9, 9], np.float32)
    got = oracle.topk(row[None], np.array([5], np.int32), 7)
    assert got[0].tolist() == [0, 1, 2, 3, 4, -1, -1]


def test_topk_negative_zero_ties_positive_zero():
    row = np.array([-0.0, 0.0, -0.0, 1.0], np.float32)
    got = oracle.topk(row[None], np.array([4], np.int32), 2)
    assert got[0].tolist() == [0, 3]


# -------------------------------------------------------------- attend ---

def test_attention_worked_example():
    fx = read_fixture("attention_worked.txt")
    q = np.array([float(v) for v in fx["q"]], np.float32).reshape(1, 1, 1, 2)
    K = np.array([[float(v) for v in fx[f"K{j}"]] for j in range(4)], np.float32)[None]
    V = np.array([[float(v) for v in fx[f"V{j}"]] for j in range(4)], np.float32)[None]
    out, lse = oracle.sparse_attn(_bf_exact(q), _bf_exact(K), _bf_exact(V),
                                  np.array([4], np.int32), np.array([[[0]]], np.int32), 4, 1.0)
    assert out[0, 0, 0].tolist() == [int(v, 16) for v in fx["expect_bits"]]
    assert lse[0, 0, 0] == np.float32(float(fx["expect_lse"][0]))


def _dense_attention(q, K, V, scale):
    z = scale * (K @ q.T)                     # [n][H]
    lse = logsumexp(z, axis=0)
    p = np.exp(z - lse[None, :])
    return (p.T @ V), lse


def test_attention_all_groups_is_dense_attention():
    spec = synth.Spec(B=1, lengths=[96], H_q=3, d_qk=32, d_v=16, seed=20)
    c = synth.generate(spec)
    G = 24
    idx = np.arange(G, dtype=np.int32)[None, None]
    out, lse = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, 4, 0.3)
    q = unbf(c["q"][0, 0]).astype(np.float64)
    K = unbf(c["K"][0]).astype(np.float64)
    V = unbf(c["V"][0]).astype(np.float64)
    ref, ref_lse = _dense_attention(q, K, V, 0.3)
    ref_bf = bf(ref.astype(np.float32))
    # both round the same real value once; allow one bf16 step where float32
    # pre-rounding of the reference lands on the other side of a midpoint
    diff = np.abs(out[0, 0].astype(np.int32) - ref_bf.astype(np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.95
    assert np.allclose(lse[0, 0], ref_lse, rtol=1e-6)


def test_attention_order_of_groups_irrelevant_and_padding_skipped():
    spec = synth.Spec(B=1, lengths=[80], H_q=2, d_qk=16, d_v=16, seed=21)
    c = synth.generate(spec)
    a = np.array([[[3, 7, 11, -1, -1]]], np.int32)
    b = np.array([[[11, -1, 3, 7, -1]]], np.int32)
    oa, la = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], a, 4, 0.25)
    ob, lb = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], b, 4, 0.25)
    assert np.array_equal(oa, ob) and np.allclose(la, lb, rtol=1e-7)


def test_attention_constant_values_and_zero_query():
    spec = synth.Spec(B=1, lengths=[64], H_q=2, d_qk=16, d_v=8, seed=22)
    c = synth.generate(spec)
    V = np.zeros_like(c["V"]); V[...] = _bf_exact(np.float32(1.75))
    idx = np.array([[[1, 4, 9]]], np.int32)
    out, _ = oracle.sparse_attn(c["q"], c["K"], V, c["seq_len"], idx, 4, 0.125)
    assert (out == _bf_exact(np.float32(1.75))).all()
    # q = 0: uniform weights -> mean of the selected value rows
    q0 = np.zeros_like(c["q"])
    out0, lse0 = oracle.sparse_attn(q0, c["K"], c["V"], c["seq_len"], idx, 4, 0.125)
    toks = [4 * g + i for g in (1, 4, 9) for i in range(4)]
    mean = unbf(c["V"][0, toks]).astype(np.float64).mean(axis=0)
    assert np.abs(unbf(out0[0, 0, 0]) - mean).max() <= 2 ** -7 * np.abs(mean).max()
    assert np.isclose(lse0[0, 0, 0], math.log(12.0), rtol=1e-7)


def test_attention_no_tokens():
    spec = synth.Spec(B=1, lengths=[16], H_q=2, d_qk=16, d_v=8, seed=23)
    c = synth.generate(spec)
    idx = np.array([[[-1, 4, 99]]], np.int32)      # padding and out-of-range only
    out, lse = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, 4, 0.125)
    assert (out == 0).all() and (lse == -np.inf).all()


# --------------------------------------------------------------- step ----

def test_retrieval_step_is_composition():
    spec = synth.Spec(B=2, lengths=[256, 200], T=3, prefill=True, H_i=4, k=7, H_q=4, d_qk=32,
                      d_v=16, seed=24)
    c = synth.generate(spec)
    r = oracle.decode_case(c)
    s = oracle.index_scores(c["q_idx"], c["w_head"], r["k_pooled"], c["seq_len"], 4, c["q_pos"])
    nv = oracle.visible_counts(c["seq_len"], c["q_pos"], 2, 3, 4)
    idx = oracle.topk(s, nv, 7)
    out, lse = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, 4, c["scale"])
    assert np.array_equal(s, r["scores"]) and np.array_equal(idx, r["idx"])
    assert np.array_equal(out, r["out"]) and np.array_equal(lse, r["lse"])
    for b in range(2):
        for t in range(3):
            assert r["idx"][b, t].tolist() == _brute_topk(s[b, t], int(nv[b, t]), 7)


def test_tiny_workload_scores_are_exact_multiples():
    # integer keys/queries, dyadic pool weights, head weights in {1/4, 1/2}:
    # every score is an exact multiple of 1/32 (exact in fp32)
    c = synth.generate(synth.named("tiny"), with_kv=False)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    s = oracle.index_scores(c["q_idx"], c["w_head"], kp, c["seq_len"], 4)[0, 0]
    ki = unbf(c["k_idx"][0]).astype(np.int64).reshape(1024, 4, 64)
    kbar8 = 4 * ki[:, 0] + 2 * ki[:, 1] + ki[:, 2] + ki[:, 3]          # 8 * kbar
    q = unbf(c["q_idx"][0, 0]).astype(np.int64)                         # [4][64]
    w4 = (c["w_head"][0, 0] * 4).astype(np.int64)                       # 4 * w
    ref32 = (np.maximum(kbar8 @ q.T, 0) * w4[None, :]).sum(axis=1)      # 32 * s
    assert np.array_equal(s.astype(np.float64) * 32, ref32.astype(np.float64))
