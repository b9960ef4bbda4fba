"""Cross-layer reuse of a selection (lcsw_decode_reuse): a later DSA layer of
the same decode step attends over the groups an earlier layer selected, with
no indexer scores or top-k of its own.  Checked against the oracle's
attention over the oracle's selection of the earlier layer."""
import numpy as np
import pytest
import torch

import long_context_sparse_weighted_b300 as lcsw
import oracle
import synth
from gpu_util import assert_attn_close, assert_lse_close, dev, dev_bf16, host_bits, upload_case

pytestmark = pytest.mark.gpu


def _layers(spec, seed2):
    """Two layers of one decode step: the same sequences (lengths), their own
    queries and caches."""
    c1 = synth.generate(spec)
    c2 = synth.generate(synth.Spec(**{**spec.__dict__, "seed": seed2}))
    return c1, c2


PATHS = [0, lcsw.FORCE_MULTIKERNEL]   # persistent kernel, split-K launches


@pytest.mark.parametrize("flags", PATHS, ids=["persistent", "split_k"])
@pytest.mark.parametrize("name,factor", [("decode_1m", 16), ("decode_b8", 16),
                                         ("ragged_b64", 32)])
def test_reuse_attends_over_the_earlier_layers_selection(name, factor, flags):
    spec = synth.shrink(synth.named(name), factor)
    c1, c2 = _layers(spec, spec.seed + 500)
    ref1 = oracle.decode_case(c1)
    d1 = upload_case(c1)
    idx = torch.empty(spec.B, spec.k, dtype=torch.int32, device="cuda")
    dec = lcsw.Decoder(d1["q_idx"][:, 0], d1["w_head"][:, 0], dev_bf16(ref1["k_pooled"]),
                       d1["q"][:, 0], d1["K"], d1["V"], d1["seq_len"], spec.P, spec.k,
                       c1["scale"], idx_out=idx)
    dec()
    dec.status()
    assert np.array_equal(idx.cpu().numpy(), ref1["idx"][:, 0])
    d2 = upload_case(c2)
    step = lcsw.ReuseStep(d2["q"][:, 0], d2["K"], d2["V"], d2["seq_len"], idx, spec.P,
                          c2["scale"], ws=dec.ws, flags=flags)
    out, lse = step()
    step.status()
    o_ref, l_ref = oracle.sparse_attn(c2["q"], c2["K"], c2["V"], c2["seq_len"], ref1["idx"],
                                      spec.P, c2["scale"])
    assert_attn_close(host_bits(out), o_ref[:, 0])
    assert_lse_close(lse.cpu().numpy(), l_ref[:, 0])


@pytest.mark.parametrize("flags", PATHS, ids=["persistent", "split_k"])
def test_reuse_skips_padding_and_out_of_range_groups(flags):
    spec = synth.Spec(B=3, lengths=[1024, 4096, 600], H_i=4, k=300, H_q=32, seed=240)
    c = synth.generate(spec)
    G = [L // 4 for L in spec.lengths]
    rng = np.random.default_rng(240)
    idx = np.full((3, 1, 300), -1, np.int32)
    for b in range(3):
        n = min(G[b], 250)
        idx[b, 0, :n] = np.sort(rng.choice(G[b], n, replace=False))
    idx[2, 0, 250] = G[2] + 7  # past the sequence: skipped like padding
    d = upload_case(c)
    step = lcsw.ReuseStep(d["q"][:, 0], d["K"], d["V"], d["seq_len"], dev(idx[:, 0]), 4,
                          c["scale"], flags=flags)
    out, lse = step()
    step.status()
    o_ref, l_ref = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, 4, c["scale"])
    assert_attn_close(host_bits(out), o_ref[:, 0])
    assert_lse_close(lse.cpu().numpy(), l_ref[:, 0])


def _random_selection(G, k, B, seed):
    """A seeded selection of k distinct groups per sequence (an input of the
    reuse step, drawn here rather than by any kernel)."""
    rng = np.random.default_rng(seed)
    idx = np.full((B, 1, k), -1, np.int32)
    for b in range(B):
        n = min(G[b], k)
        idx[b, 0, :n] = rng.choice(G[b], n, replace=False)
    return idx


def test_reuse_repeated_calls_leave_the_workspace_ready():
    """The persistent path clears the partial words it read: a second call on
    the same workspace gives the same bits."""
    spec = synth.Spec(B=2, lengths=[20000, 9000], H_i=4, k=512, H_q=64, seed=241)
    c = synth.generate(spec)
    idx = _random_selection([L // 4 for L in spec.lengths], spec.k, spec.B, 241)
    d = upload_case(c)
    step = lcsw.ReuseStep(d["q"][:, 0], d["K"], d["V"], d["seq_len"], dev(idx[:, 0]), 4,
                          c["scale"])
    o1 = step()[0].clone()
    step.status()
    o2, lse = step()
    step.status()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    o_ref, l_ref = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, 4, c["scale"])
    assert_attn_close(host_bits(o2), o_ref[:, 0])
    assert_lse_close(lse.cpu().numpy(), l_ref[:, 0])


@pytest.mark.slow
def test_reuse_full_size_decode_1m():
    """The benchmarked reuse call: decode_1m's full cache (1,048,576 tokens),
    64 query heads, 512 groups drawn by a seeded generator."""
    spec = synth.named("decode_1m")
    c = synth.generate(synth.Spec(**{**spec.__dict__, "seed": spec.seed + 500}))
    idx = _random_selection([L // 4 for L in spec.lengths], spec.k, spec.B, 242)
    d = upload_case(c)
    step = lcsw.ReuseStep(d["q"][:, 0], d["K"], d["V"], d["seq_len"], dev(idx[:, 0]), spec.P,
                          c["scale"])
    out, lse = step()
    step.status()
    o_ref, l_ref = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, spec.P,
                                      c["scale"])
    assert_attn_close(host_bits(out), o_ref[:, 0])
    assert_lse_close(lse.cpu().numpy(), l_ref[:, 0])
