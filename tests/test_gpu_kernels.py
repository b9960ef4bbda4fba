"""Per-kernel parity of liblcsw (through the C ABI) against the CPU oracle.

Every input comes from synth (seeded) or from the oracle; nothing the CUDA
path produced is ever fed to the oracle or used as an expected value.
"""
import numpy as np
import pytest
import torch

import long_context_sparse_weighted_b300 as lcsw
import oracle
import synth
from gpu_util import (assert_attn_close, assert_lse_close, assert_scores_close, dev, dev_bf16,
                      host_bits, upload_case)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    lcsw.lib()


# ------------------------------------------------------------------ pool ---

@pytest.mark.parametrize("P", [1, 2, 4, 8])
@pytest.mark.parametrize("mode", ["softmax", "dyadic", "random"])
def test_pool_keys_bit_exact(P, mode):
    spec = synth.Spec(B=3, lengths=[P * 333 + P - 1, 4096, 40], L_cap=4104, P=P, pool_mode=mode,
                      seed=100 + P)
    c = synth.generate(spec, with_kv=False)
    ref = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], P)
    d = upload_case(c)
    out = torch.full((spec.B, spec.G_max, 64), 0x1357, dtype=torch.int16, device="cuda")
    sentinel = host_bits(out.clone())
    lcsw.pool_keys(d["k_idx"], d["pool_w"], d["seq_len"], P, out.view(torch.bfloat16))
    got = host_bits(out)
    for b, L in enumerate(spec.lengths):
        G = L // P
        assert np.array_equal(got[b, :G], ref[b, :G]), f"b={b}"
        assert np.array_equal(got[b, G:], sentinel[b, G:]), "rows past the last group changed"


def test_pool_keys_hard_sums_bit_exact():
    """Sums on or a hair beside a bf16 midpoint, after cancellation of large
    terms, or spanning hundreds of binades (tests/pool_cases.py): the kernel
    and the exact oracle agree bit for bit, and both equal the nearest bf16 of
    the exact rational sum."""
    import pool_cases
    cs = pool_cases.cases(n=800, seed=32)
    k_idx, pool_w = pool_cases.as_arrays(cs)
    seq = np.array([k_idx.shape[1]], np.int32)
    ref = oracle.pool_keys(k_idx, pool_w, seq, 4)
    for g, (a, k) in enumerate(cs[:64]):
        assert ref[0, g, 0] == pool_cases.round_bf16(pool_cases.exact_sum(a, k))
    out = torch.zeros(1, len(cs), 64, dtype=torch.bfloat16, device="cuda")
    lcsw.pool_keys(dev_bf16(k_idx), dev(pool_w), dev(seq), 4, out)
    got = host_bits(out)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} elements differ, first groups {sorted(set(bad[:, 1]))[:8]}"


def test_pool_keys_tiny_workload_exact():
    c = synth.generate(synth.named("tiny"), with_kv=False)
    ref = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    d = upload_case(c)
    out = torch.zeros(1, c["G_max"], 64, dtype=torch.bfloat16, device="cuda")
    lcsw.pool_keys(d["k_idx"], d["pool_w"], d["seq_len"], 4, out)
    assert np.array_equal(host_bits(out), ref)


def test_pool_keys_group_window_and_strides():
    spec = synth.Spec(B=2, lengths=[400, 256], L_cap=512, P=4, seed=103)
    c = synth.generate(spec, with_kv=False)
    ref = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    d = upload_case(c)
    big = torch.zeros(2, 200, 64, dtype=torch.bfloat16, device="cuda")   # capacity > G_max
    view = big[:, :128]
    g_begin = dev(np.array([90, 10], np.int32))
    lcsw.pool_keys(d["k_idx"], d["pool_w"], d["seq_len"], 4, view, g_begin=g_begin, g_span=20)
    got = host_bits(big)
    assert np.array_equal(got[0, 90:100], ref[0, 90:100])      # clipped at G = 100
    assert np.array_equal(got[1, 10:30], ref[1, 10:30])
    assert (got[0, :90] == 0).all() and (got[1, 30:] == 0).all() and (got[1, :10] == 0).all()


# ---------------------------------------------------------------- scores ---

def test_scores_tiny_workload_bit_exact():
    c = synth.generate(synth.named("tiny"), with_kv=False)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    ref = oracle.index_scores(c["q_idx"], c["w_head"], kp, c["seq_len"], 4)
    d = upload_case(c)
    got = lcsw.index_scores(d["q_idx"], d["w_head"], dev_bf16(kp), d["seq_len"], 4).cpu().numpy()
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("H_i", [1, 3, 8, 12, 16])
def test_scores_gaussian_within_tolerance(H_i):
    spec = synth.Spec(B=2, lengths=[8196, 1000], H_i=H_i, seed=110 + H_i)
    c = synth.generate(spec, with_kv=False)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    ref = oracle.index_scores(c["q_idx"], c["w_head"], kp, c["seq_len"], 4)
    d = upload_case(c)
    got = lcsw.index_scores(d["q_idx"], d["w_head"], dev_bf16(kp), d["seq_len"], 4).cpu().numpy()
    assert_scores_close(got, ref)


@pytest.mark.parametrize("T", [2, 5, 9])
def test_scores_causal_multi_query(T):
    spec = synth.Spec(B=2, lengths=[4000, 1203], T=T, prefill=True, w_mode="signed",
                      seed=120 + T)
    c = synth.generate(spec, with_kv=False)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    ref = oracle.index_scores(c["q_idx"], c["w_head"], kp, c["seq_len"], 4, q_pos=c["q_pos"])
    d = upload_case(c)
    got = lcsw.index_scores(d["q_idx"], d["w_head"], dev_bf16(kp), d["seq_len"], 4,
                            q_pos=d["q_pos"]).cpu().numpy()
    assert_scores_close(got, ref)


# Prefill query blocks (T >= 64) score on the tcgen05 GEMM: tiles of 128 queries
# x 128 groups, ragged in both directions; G_max % 4 != 0 takes the scalar
# store path.
@pytest.mark.parametrize("H_i,T,L0,L1", [(8, 300, 16012, 9001), (1, 128, 4096, 777),
                                         (16, 77, 10004, 5000)])
def test_scores_tensor_core_prefill(H_i, T, L0, L1):
    spec = synth.Spec(B=2, lengths=[L0, L1], T=T, prefill=True, H_i=H_i, w_mode="signed",
                      seed=140 + H_i)
    c = synth.generate(spec, with_kv=False)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    ref = oracle.index_scores(c["q_idx"], c["w_head"], kp, c["seq_len"], 4, q_pos=c["q_pos"])
    d = upload_case(c)
    got = lcsw.index_scores(d["q_idx"], d["w_head"], dev_bf16(kp), d["seq_len"], 4,
                            q_pos=d["q_pos"]).cpu().numpy()
    assert_scores_close(got, ref)


def test_scores_tensor_core_exact_integer_inputs():
    # integer-valued keys and queries, dyadic pooling and head weights: every
    # product and sum is exact in fp32, so the GEMM path is bit-exact
    spec = synth.Spec(B=1, lengths=[4096 + 200], T=200, prefill=True, H_i=4, idx_values="int3",
                      w_mode="quarter_half", pool_mode="dyadic", seed=130)
    c = synth.generate(spec, with_kv=False)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4)
    ref = oracle.index_scores(c["q_idx"], c["w_head"], kp, c["seq_len"], 4, q_pos=c["q_pos"])
    d = upload_case(c)
    got = lcsw.index_scores(d["q_idx"], d["w_head"], dev_bf16(kp), d["seq_len"], 4,
                            q_pos=d["q_pos"]).cpu().numpy()
    assert np.array_equal(got, ref)


def test_visible_counts_exact():
    seq = np.array([0, 3, 4, 17, 4096], np.int32)
    q_pos = np.array([[-1, 0, 2], [0, 1, 2], [2, 3, 3], [3, 7, 16], [100, 4094, 4095]], np.int32)
    ref = oracle.visible_counts(seq, q_pos, 5, 3, 4)
    got = lcsw.visible_counts(dev(seq), dev(q_pos), 5, 3, 4).cpu().numpy()
    assert np.array_equal(got, ref)
    ref0 = oracle.visible_counts(seq, None, 5, 1, 4)
    got0 = lcsw.visible_counts(dev(seq), None, 5, 1, 4).cpu().numpy()
    assert np.array_equal(got0, ref0)


# ------------------------------------------------------------------ top-k ---

def _topk_case(rows, G, kind, seed):
    rng = np.random.default_rng(seed)
    if kind == "ties":
        s = rng.integers(-3, 4, size=(rows, G)).astype(np.float32)
    elif kind == "zeros":
        s = np.zeros((rows, G), np.float32)
        s[:, ::3] = -0.0
    elif kind == "wide":
        s = (rng.standard_normal((rows, G)) * np.exp(rng.uniform(-20, 20, (rows, G)))).astype(np.float32)
    else:
        s = rng.standard_normal((rows, G)).astype(np.float32) * 10
    return s


@pytest.mark.parametrize("kind", ["normal", "ties", "zeros", "wide"])
@pytest.mark.parametrize("k", [1, 64, 512])
def test_topk_bit_exact_on_oracle_scores(kind, k):
    rows, G = 6, 5000
    s = _topk_case(rows, G, kind, 130 + k)
    n_valid = np.array([5000, 4999, 700, k, k - 1 if k > 1 else 0, 0], np.int32)
    ref = oracle.topk(s, n_valid, k)
    got = lcsw.topk_groups(dev(s), dev(n_valid), k).cpu().numpy()
    assert np.array_equal(got, ref)


def test_topk_long_row():
    s = _topk_case(1, 262144, "normal", 140)
    s[0, 1000:1010] = s.max()          # ties at the top
    n_valid = np.array([262144], np.int32)
    ref = oracle.topk(s, n_valid, 512)
    got = lcsw.topk_groups(dev(s), dev(n_valid), 512).cpu().numpy()
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("case", ["normal", "ties_at_k", "all_equal", "short_rows",
                                  "one_hot_digit"])
def test_topk_few_long_rows_multi_block(case):
    """Few long rows take the multi-block selection (histogram, filter,
    final); each must equal the oracle bit for bit.  all_equal overflows the
    candidate list and takes the one-block fallback inside the last launch;
    short_rows mixes rows with n_valid <= k and a row below the list's size."""
    rows, G, k = 4, 262144, 512
    s = _topk_case(rows, G, "normal", 150)
    n_valid = np.array([G, G - 3, 200000, 131073], np.int32)
    if case == "ties_at_k":
        s[:, 5000:9000] = np.sort(s[0])[-400]       # a wide tie around the k-th score
    elif case == "all_equal":
        s[1] = 0.75
        s[2, :] = -0.0
        s[2, ::7] = 0.0                             # -0 and +0 tie
    elif case == "short_rows":
        n_valid = np.array([G, 300, 512, 20000], np.int32)
    elif case == "one_hot_digit":
        s[3] = np.float32(1.0) + np.arange(G, dtype=np.float32) * np.float32(2 ** -23)
    assert lcsw.lib().lcsw_topk_workspace_size(rows, G, k) > 0
    ref = oracle.topk(s, n_valid, k)
    got = lcsw.topk_groups(dev(s), dev(n_valid), k).cpu().numpy()
    assert np.array_equal(got, ref)


# -------------------------------------------------------------- attention ---

def _attn_case(B, lengths, T, H_q, d_qk, d_v, k, P, seed, pad=0):
    spec = synth.Spec(B=B, lengths=lengths, T=T, H_q=H_q, d_qk=d_qk, d_v=d_v, P=P, k=k,
                      seed=seed)
    c = synth.generate(spec)
    rng = np.random.default_rng(seed)
    idx = np.full((B, T, k), -1, np.int32)
    for b in range(B):
        G = lengths[b] // P
        for t in range(T):
            n = min(k - pad, G)
            idx[b, t, :n] = np.sort(rng.choice(G, size=n, replace=False))
    return c, idx


@pytest.mark.parametrize("H_q,d_qk,d_v", [(16, 128, 128), (32, 192, 128), (64, 128, 128),
                                          (128, 128, 128), (32, 64, 64), (16, 128, 64)])
def test_sparse_attn_shapes(H_q, d_qk, d_v):
    c, idx = _attn_case(2, [4096, 1500], 1, H_q, d_qk, d_v, 100, 4, 150 + H_q + d_qk, pad=3)
    out_r, lse_r = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, 4, c["scale"])
    d = upload_case(c)
    out, lse = lcsw.sparse_attn(d["q"], d["K"], d["V"], d["seq_len"], dev(idx), 4, c["scale"])
    assert_attn_close(host_bits(out), out_r)
    assert_lse_close(lse.cpu().numpy(), lse_r)


@pytest.mark.parametrize("P", [1, 2, 8])
def test_sparse_attn_pool_sizes(P):
    c, idx = _attn_case(1, [8192], 1, 32, 128, 128, 2048 // P, P, 160 + P)
    out_r, lse_r = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, P, c["scale"])
    d = upload_case(c)
    out, lse = lcsw.sparse_attn(d["q"], d["K"], d["V"], d["seq_len"], dev(idx), P, c["scale"])
    assert_attn_close(host_bits(out), out_r)
    assert_lse_close(lse.cpu().numpy(), lse_r)


def test_sparse_attn_many_rows_single_split():
    c, idx = _attn_case(2, [2048, 3000], 160, 32, 128, 128, 40, 4, 170)
    out_r, lse_r = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, 4, c["scale"])
    d = upload_case(c)
    out, lse = lcsw.sparse_attn(d["q"], d["K"], d["V"], d["seq_len"], dev(idx), 4, c["scale"])
    assert_attn_close(host_bits(out), out_r)
    assert_lse_close(lse.cpu().numpy(), lse_r)


def test_sparse_attn_empty_and_out_of_range():
    c, idx = _attn_case(2, [256, 256], 1, 16, 128, 128, 8, 4, 180)
    idx[0, 0, :] = -1                   # nothing selected
    idx[1, 0, :] = [0, 5, 63, 64, 1000, -7, 70, 2]   # 64, 1000, -7, 70 are out of range
    out_r, lse_r = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, 4, c["scale"])
    d = upload_case(c)
    out, lse = lcsw.sparse_attn(d["q"], d["K"], d["V"], d["seq_len"], dev(idx), 4, c["scale"])
    got = host_bits(out)
    assert (got[0] == 0).all() and np.isneginf(lse.cpu().numpy()[0]).all()
    assert_attn_close(got[1:], out_r[1:])
    assert_lse_close(lse.cpu().numpy(), lse_r)
