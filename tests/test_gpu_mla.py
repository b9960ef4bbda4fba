"""The MLA latent geometry on the GPU against the oracle.

One 576-wide row per token (latent 512 + rotary 64) serves as the key, and its
first 512 dims as the value.  The oracle's attention is the plain definition
with K = the rows and V = their latent part (a copy), so it knows nothing of
the sharing; the kernel reads each row once.  Tolerances as for the other
attention paths (tests/gpu_util.py).
"""
import numpy as np
import pytest
import torch

import long_context_sparse_weighted_b300 as lcsw
import oracle
import synth
from gpu_util import assert_attn_close, assert_lse_close, dev, dev_bf16, host_bits, upload_case

pytestmark = pytest.mark.gpu


def _mla_spec(**kw):
    base = dict(B=2, lengths=[6000, 3000], H_i=4, k=128, H_q=32, d_qk=576, d_v=512, mla=True,
                seed=300)
    base.update(kw)
    return synth.Spec(**base)


def _selection(G, k, B, T, seed, pad_invalid=True):
    """Seeded selections: k distinct groups per row, -1 padded; one entry past
    the sequence where there is room (skipped like padding)."""
    rng = np.random.default_rng(seed)
    idx = np.full((B, T, k), -1, np.int32)
    for b in range(B):
        for t in range(T):
            n = min(G[b], k - 1)
            idx[b, t, :n] = np.sort(rng.choice(G[b], n, replace=False))
            if pad_invalid:
                idx[b, t, n] = G[b] + 3
    return idx


@pytest.mark.parametrize("B,T,H_q,lengths,k", [
    (2, 1, 32, [6000, 3000], 128),
    (1, 1, 64, [20000], 512),
    (3, 2, 16, [1024, 4096, 700], 64),
    (1, 1, 64, [256], 512),            # fewer groups than k: padding throughout
])
def test_mla_attention_matches_oracle(B, T, H_q, lengths, k):
    spec = _mla_spec(B=B, T=T, H_q=H_q, lengths=lengths, k=k, seed=300 + B + H_q)
    c = synth.generate(spec)
    idx = _selection([L // 4 for L in lengths], k, B, T, spec.seed)
    o_ref, l_ref = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, 4, c["scale"])
    out, lse = lcsw.sparse_attn_mla(dev_bf16(c["q"]), dev_bf16(c["K"]), dev(c["seq_len"]),
                                    dev(idx), 4, c["scale"])
    torch.cuda.synchronize()
    assert_attn_close(host_bits(out), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)


@pytest.mark.parametrize("flags", [0, lcsw.FORCE_MULTIKERNEL], ids=["fused_select", "launches"])
def test_mla_decode_step_selects_and_attends_like_the_oracle(flags):
    """lcsw_decode_fused in the MLA geometry (V = NULL): the indexer selection
    bit for bit, then attention over the latent rows.  By default the
    persistent kernel selects (its attention skipped) and the latent attention
    follows; the forced path runs scores, top-k and attention as separate
    launches."""
    spec = _mla_spec(B=2, lengths=[40000, 12000], H_i=8, k=256, H_q=64, seed=310)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    d = upload_case(c)
    idx = torch.empty(spec.B, spec.k, dtype=torch.int32, device="cuda")
    dec = lcsw.Decoder(d["q_idx"][:, 0], d["w_head"][:, 0], dev_bf16(ref["k_pooled"]),
                       d["q"][:, 0], d["K"], None, d["seq_len"], spec.P, spec.k, c["scale"],
                       idx_out=idx, flags=flags)
    merge = 1 if lcsw.lib().lcsw_sparse_attn_mla_workspace_size(spec.B, 1, spec.H_q, spec.k, 4) else 0
    topk = 3 if lcsw.lib().lcsw_topk_workspace_size(spec.B, spec.G_max, spec.k) else 1
    assert dec.launches_per_call == (2 if flags == 0 else 2 + topk) + merge
    out, lse = dec()
    dec.status()
    assert np.array_equal(idx.cpu().numpy(), ref["idx"][:, 0])
    assert_attn_close(host_bits(out), ref["out"][:, 0])
    assert_lse_close(lse.cpu().numpy(), ref["lse"][:, 0])


def test_mla_reuse_step():
    spec = _mla_spec(B=2, lengths=[9000, 30000], k=200, H_q=32, seed=320)
    c = synth.generate(spec)
    idx = _selection([L // 4 for L in spec.lengths], spec.k, spec.B, 1, 320)
    d = upload_case(c)
    step = lcsw.ReuseStep(d["q"][:, 0], d["K"], None, d["seq_len"], dev(idx[:, 0]), 4,
                          c["scale"])
    out, lse = step()
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, 4, c["scale"])
    assert_attn_close(host_bits(out), o_ref[:, 0])
    assert_lse_close(lse.cpu().numpy(), l_ref[:, 0])


def test_mla_rejects_a_separate_value_cache():
    spec = _mla_spec(B=1, lengths=[2048], k=16, H_q=16, seed=330)
    c = synth.generate(spec)
    d = upload_case(c)
    with pytest.raises(lcsw.LcswError):
        dec = lcsw.Decoder(d["q_idx"][:, 0], d["w_head"][:, 0], dev_bf16(np.zeros(
            (1, spec.G_max, 64), np.uint16)), d["q"][:, 0], d["K"],
            torch.zeros(1, spec.L_max, 512, dtype=torch.bfloat16, device="cuda"), d["seq_len"],
            4, spec.k, c["scale"])
        dec()


@pytest.mark.slow
def test_mla_attention_full_size_decode_1m():
    """The benchmarked MLA attention call: decode_1m's 1,048,576-token latent
    cache, 64 heads, 512 groups drawn by a seeded generator."""
    spec = synth.named("mla_decode_1m")
    c = synth.generate(spec)
    idx = _selection([L // 4 for L in spec.lengths], spec.k, 1, 1, 340, pad_invalid=False)
    o_ref, l_ref = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, 4, c["scale"])
    out, lse = lcsw.sparse_attn_mla(dev_bf16(c["q"]), dev_bf16(c["K"]), dev(c["seq_len"]),
                                    dev(idx), 4, c["scale"])
    torch.cuda.synchronize()
    assert_attn_close(host_bits(out), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)


@pytest.mark.slow
def test_mla_decode_step_full_size():
    """The benchmarked MLA decode step: decode_1m's indexer and selection over
    1,048,576 tokens, attention over the 576-wide latent rows, against the
    oracle's whole step (pool, score, top-k, attention)."""
    spec = synth.named("mla_decode_1m")
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    d = upload_case(c)
    kp = dev_bf16(ref["k_pooled"]).clone()
    kp[0, -1] = 0  # the step re-pools the newest group itself
    idx = torch.empty(spec.B, spec.k, dtype=torch.int32, device="cuda")
    dec = lcsw.Decoder(d["q_idx"][:, 0], d["w_head"][:, 0], kp, d["q"][:, 0], d["K"], None,
                       d["seq_len"], spec.P, spec.k, c["scale"], k_idx=d["k_idx"],
                       pool_w=d["pool_w"], idx_out=idx)
    out, lse = dec()
    dec.status()
    assert np.array_equal(idx.cpu().numpy(), ref["idx"][:, 0])
    assert_attn_close(host_bits(out), ref["out"][:, 0])
    assert_lse_close(lse.cpu().numpy(), ref["lse"][:, 0])


@pytest.mark.parametrize("P", [1, 2, 8])
def test_mla_attention_other_pool_sizes(P):
    """Groups of 1, 2 and 8 latent rows (64/P groups a chunk), two sequences
    whose lengths are not multiples of P."""
    lengths = [7001, 2999]
    spec = _mla_spec(B=2, lengths=lengths, H_q=32, k=96, P=P, seed=350 + P)
    c = synth.generate(spec)
    idx = _selection([L // P for L in lengths], spec.k, 2, 1, spec.seed)
    o_ref, l_ref = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, P, c["scale"])
    out, lse = lcsw.sparse_attn_mla(dev_bf16(c["q"]), dev_bf16(c["K"]), dev(c["seq_len"]),
                                    dev(idx), P, c["scale"])
    torch.cuda.synchronize()
    assert_attn_close(host_bits(out), o_ref)
    assert_lse_close(lse.cpu().numpy(), l_ref)
