"""INT8 K/V cache on the GPU against the oracle's INT8 attention.

The row quantizer must give the oracle's codes and scales bit for bit; the
attention over the codes must match oracle.sparse_attn_i8kv within the
attention tolerances (tests/gpu_util.py).  The oracle quantizes the bf16 rows
itself: nothing it reads comes from the GPU.
"""
import numpy as np
import pytest
import torch

import long_context_sparse_weighted_b300 as lcsw
import oracle
import synth
from gpu_util import assert_attn_close, assert_lse_close, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("width", [64, 128, 192])
def test_quantize_rows_i8_bit_exact(width):
    rng = np.random.default_rng(600 + width)
    B, L = 2, 300
    x = rng.standard_normal((B, L, width)).astype(np.float32)
    x[0, 0] = 0.0                                   # zero row: scale 0, codes 0
    x[0, 1] *= 1e-37                                # scale in the fp32 subnormals
    x[1, 2] *= 1e30
    x[1, 3, :] = np.round(np.linspace(-127.0, 127.0, width))  # scale 1: the codes themselves
    x[1, 4, :] = (np.arange(width) % 8 - 4) + 0.5   # halves at scale 1 (127 sets the amax)
    x[1, 4, 0] = 127.0
    xb = synth.bf16_bits(x)
    codes, scales = oracle.quantize_rows_i8(xb)
    gc, gs = lcsw.quantize_rows_i8(dev_bf16(xb))
    torch.cuda.synchronize()
    assert np.array_equal(gs.cpu().numpy().view(np.uint32), scales.view(np.uint32))
    bad = np.argwhere(gc.cpu().numpy() != codes)
    assert bad.size == 0, f"{len(bad)} codes differ, e.g. {bad[:4].tolist()}"


def test_quantize_rows_i8_window_writes_only_its_rows():
    rng = np.random.default_rng(610)
    B, L, W = 3, 64, 128
    xb = synth.bf16_bits(rng.standard_normal((B, L, W)).astype(np.float32))
    codes = torch.full((B, L, W), 99, dtype=torch.int8, device="cuda")
    scales = torch.full((B, L), -1.0, dtype=torch.float32, device="cuda")
    rb = np.array([5, 0, 60], np.int32)
    lcsw.quantize_rows_i8(dev_bf16(xb), codes, scales, row_begin=dev(rb), n_rows=3)
    torch.cuda.synchronize()
    oc, os_ = oracle.quantize_rows_i8(xb)
    gc, gs = codes.cpu().numpy(), scales.cpu().numpy()
    for b in range(B):
        inside = np.zeros(L, bool)
        inside[rb[b]:rb[b] + 3] = True
        assert np.array_equal(gc[b, inside], oc[b, inside])
        assert np.array_equal(gs[b, inside].view(np.uint32), os_[b, inside].view(np.uint32))
        assert (gc[b, ~inside] == 99).all() and (gs[b, ~inside] == -1.0).all()


def _selection(G, k, B, T, seed):
    rng = np.random.default_rng(seed)
    idx = np.full((B, T, k), -1, np.int32)
    for b in range(B):
        for t in range(T):
            n = min(G[b], k - 1)
            idx[b, t, :n] = np.sort(rng.choice(G[b], n, replace=False))
            idx[b, t, -1] = G[b] + 2                 # past the sequence: skipped
    return idx


@pytest.mark.parametrize("H_q,d_qk,d_v,T", [(16, 128, 128, 1), (32, 192, 128, 1),
                                            (64, 128, 128, 1), (32, 128, 64, 3),
                                            (16, 64, 64, 2)])
def test_kvi8_attention_matches_oracle(H_q, d_qk, d_v, T):
    lengths = [9000, 2500]
    spec = synth.Spec(B=2, lengths=lengths, T=T, H_q=H_q, d_qk=d_qk, d_v=d_v, k=200,
                      seed=620 + H_q + d_qk)
    c = synth.generate(spec)
    kc, ks = oracle.quantize_rows_i8(c["K"])
    vc, vs = oracle.quantize_rows_i8(c["V"])
    idx = _selection([L // 4 for L in lengths], spec.k, spec.B, T, spec.seed)
    o_ref, l_ref = oracle.sparse_attn_i8kv(c["q"], kc, ks, vc, vs, c["seq_len"], idx, 4,
                                           c["scale"])
    # the GPU quantizes the bf16 caches itself (bit-exact per the test above)
    gkc, gks = lcsw.quantize_rows_i8(dev_bf16(c["K"]))
    gvc, gvs = lcsw.quantize_rows_i8(dev_bf16(c["V"]))
    out, lse = lcsw.sparse_attn_kvi8(dev_bf16(c["q"]), gkc, gks, gvc, gvs, dev(c["seq_len"]),
                                     dev(idx), 4, c["scale"])
    torch.cuda.synchronize()
    assert_attn_close(host_bits(out), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)


@pytest.mark.slow
def test_kvi8_attention_full_size_decode_1m():
    """decode_1m's 1,048,576-token K/V cache in INT8, 64 heads, 512 seeded
    groups: the oracle quantizes (itself) only the rows the groups cover."""
    spec = synth.named("decode_1m")
    c = synth.generate(spec)
    G = spec.lengths[0] // 4
    rng = np.random.default_rng(630)
    groups = np.sort(rng.choice(G, spec.k, replace=False)).astype(np.int32)
    idx = groups.reshape(1, 1, spec.k)
    toks = (groups[:, None] * 4 + np.arange(4)).reshape(-1)
    kc = np.zeros((1, spec.L_max, spec.d_qk), np.int8)
    vc = np.zeros((1, spec.L_max, spec.d_v), np.int8)
    ks = np.zeros((1, spec.L_max), np.float32)
    vs = np.zeros((1, spec.L_max), np.float32)
    kc[0, toks], ks[0, toks] = oracle.quantize_rows_i8(c["K"][0, toks])
    vc[0, toks], vs[0, toks] = oracle.quantize_rows_i8(c["V"][0, toks])
    o_ref, l_ref = oracle.sparse_attn_i8kv(c["q"], kc, ks, vc, vs, c["seq_len"], idx, 4,
                                           c["scale"])
    gkc, gks = lcsw.quantize_rows_i8(dev_bf16(c["K"]))
    gvc, gvs = lcsw.quantize_rows_i8(dev_bf16(c["V"]))
    out, lse = lcsw.sparse_attn_kvi8(dev_bf16(c["q"]), gkc, gks, gvc, gvs, dev(c["seq_len"]),
                                     dev(idx), 4, c["scale"])
    torch.cuda.synchronize()
    assert_attn_close(host_bits(out), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)


@pytest.mark.parametrize("P", [1, 2, 8])
@pytest.mark.parametrize("fmt", ["i8", "e4m3"])
def test_quantized_kv_attention_other_pool_sizes(P, fmt):
    """Groups of 1, 2 and 8 tokens (a chunk holds 64/P groups), both code
    formats, a ragged pair of sequences whose lengths are not multiples of P."""
    lengths = [5003, 1201]
    spec = synth.Spec(B=2, lengths=lengths, H_q=32, d_qk=128, d_v=128, k=100, P=P,
                      seed=640 + P)
    c = synth.generate(spec)
    quant_o = oracle.quantize_rows_i8 if fmt == "i8" else oracle.quantize_rows_e4m3
    attn_o = oracle.sparse_attn_i8kv if fmt == "i8" else oracle.sparse_attn_e4m3kv
    quant_g = lcsw.quantize_rows_i8 if fmt == "i8" else lcsw.quantize_rows_e4m3
    attn_g = lcsw.sparse_attn_kvi8 if fmt == "i8" else lcsw.sparse_attn_kv8
    kc, ks = quant_o(c["K"])
    vc, vs = quant_o(c["V"])
    idx = _selection([L // P for L in lengths], spec.k, spec.B, 1, spec.seed)
    o_ref, l_ref = attn_o(c["q"], kc, ks, vc, vs, c["seq_len"], idx, P, c["scale"])
    gkc, gks = quant_g(dev_bf16(c["K"]))
    gvc, gvs = quant_g(dev_bf16(c["V"]))
    out, lse = attn_g(dev_bf16(c["q"]), gkc, gks, gvc, gvs, dev(c["seq_len"]), dev(idx), P,
                      c["scale"])
    torch.cuda.synchronize()
    assert_attn_close(host_bits(out), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)
