"""Whole decode step (lcsw_decode_fused) and chunked prefill (lcsw_prefill)
against the CPU oracle, on the named workloads (shrunk where the full size is
covered by test_gpu_fullsize.py) and on edge cases."""
import numpy as np
import pytest
import torch

import long_context_sparse_weighted_b300 as lcsw
import oracle
import synth
from gpu_util import (assert_attn_close, assert_lse_close, assert_scores_close, dev, dev_bf16,
                      host_bits, selection_diff, upload_case)

pytestmark = pytest.mark.gpu


def run_decode(c, kp, append=False, corrupt_last=False, flags=0):
    """Upload one generated decode workload and run the fused step."""
    d = upload_case(c)
    B, G_max, k = c["B"], c["G_max"], c["k"]
    kp_dev = dev_bf16(kp).clone()
    if corrupt_last:
        for b in range(B):
            G = int(c["seq_len"][b]) // c["P"]
            if G:
                kp_dev[b, G - 1] = 7.0
    idx = torch.empty(B, k, dtype=torch.int32, device="cuda")
    scores = torch.empty(B, G_max, dtype=torch.float32, device="cuda")
    kw = dict(idx_out=idx, scores_out=scores, flags=flags)
    if append:
        kw.update(k_idx=d["k_idx"], pool_w=d["pool_w"])
    dec = lcsw.Decoder(d["q_idx"][:, 0], d["w_head"][:, 0], kp_dev, d["q"][:, 0], d["K"], d["V"],
                       d["seq_len"], c["P"], k, c["scale"], **kw)
    out, lse = dec()
    dec.status()
    return dict(out=host_bits(out), lse=lse.cpu().numpy(), idx=idx.cpu().numpy(),
                scores=scores.cpu().numpy(), k_pooled=host_bits(kp_dev),
                launches=dec.launches_per_call)


def check_against_oracle(c, got, ref, exact=False):
    if exact:
        assert np.array_equal(got["scores"], ref["scores"][:, 0])
        assert np.array_equal(got["idx"], ref["idx"][:, 0])
    else:
        assert_scores_close(got["scores"], ref["scores"][:, 0])
        nd = selection_diff(got["idx"], ref["idx"][:, 0], ref["scores"][:, 0])
        assert nd == 0, f"{nd} rows selected a different (near-tie) set"
    assert_attn_close(got["out"], ref["out"][:, 0])
    assert_lse_close(got["lse"], ref["lse"][:, 0])


def test_decode_tiny_bit_exact_selection():
    c = synth.generate(synth.named("tiny"))
    ref = oracle.decode_case(c)
    got = run_decode(c, ref["k_pooled"])
    check_against_oracle(c, got, ref, exact=True)


@pytest.mark.parametrize("name,factor", [("decode_b8", 16), ("decode_1m", 32),
                                         ("ragged_b64", 32)])
def test_decode_workloads_shrunk(name, factor):
    spec = synth.shrink(synth.named(name), factor)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    got = run_decode(c, ref["k_pooled"])
    check_against_oracle(c, got, ref)


PATHS = {"persistent": 0, "persistent_multipass_select": lcsw.FORCE_MULTIPASS_SELECT,
         "multikernel": lcsw.FORCE_MULTIKERNEL}


@pytest.mark.parametrize("path", sorted(PATHS))
def test_decode_every_path_matches_oracle(path):
    spec = synth.Spec(B=3, lengths=[40000, 9000, 123456 // 4 * 4], H_i=8, k=512, H_q=64,
                      plant_frac=0.05, seed=205)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    got = run_decode(c, ref["k_pooled"], append=True, corrupt_last=True, flags=PATHS[path])
    assert (got["launches"] == 1) == (path != "multikernel")
    assert np.array_equal(got["k_pooled"], ref["k_pooled"])
    check_against_oracle(c, got, ref)


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("G", [3000, 20000])
def test_decode_all_scores_tied(path, G):
    # zero indexer queries: every score is +0, so the top k are groups 0..k-1
    spec = synth.Spec(B=1, lengths=[4 * G], H_i=4, k=300, H_q=16, seed=206)
    c = synth.generate(spec)
    c["q_idx"][:] = 0
    ref = oracle.decode_case(c)
    assert (ref["idx"][0, 0] == np.arange(300)).all()
    got = run_decode(c, ref["k_pooled"], flags=PATHS[path])
    assert np.array_equal(got["idx"], ref["idx"][:, 0])
    check_against_oracle(c, got, ref, exact=True)


@pytest.mark.parametrize("path", ["persistent", "persistent_multipass_select"])
def test_decode_one_block_sequences_past_9216_groups(path):
    """76 equal sequences of 9,250 groups: the even split gives 72 of them two
    blocks and 4 one block, whose 9,250 scores run past entry 9,216 of the
    scores kept in shared memory.  The prefetch of a block's first
    candidates (K/V rows and group ids) must leave every score alone: the
    multi-pass selection reads them all after it."""
    spec = synth.Spec(B=76, lengths=[37000] * 76, H_i=4, k=512, H_q=16, seed=209)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    got = run_decode(c, ref["k_pooled"], flags=PATHS[path])
    check_against_oracle(c, got, ref)


def test_decode_bounded_wait_reports_timeout():
    """A block that never arrives at a cross-block barrier: the other blocks'
    bounded waits run out, the call returns, and the status reads TIMEOUT."""
    spec = synth.Spec(B=1, lengths=[65536], H_i=8, k=64, H_q=16, seed=207)
    c = synth.generate(spec)
    d = upload_case(c)
    kp = dev_bf16(oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], 4))
    dec = lcsw.Decoder(d["q_idx"][:, 0], d["w_head"][:, 0], kp, d["q"][:, 0], d["K"], d["V"],
                       d["seq_len"], 4, 64, c["scale"], flags=lcsw.TEST_SKIP_ARRIVE)
    assert dec.launches_per_call == 1
    dec()
    with pytest.raises(lcsw.LcswError) as ei:
        dec.status()
    assert ei.value.status == lcsw.ERR_TIMEOUT
    # the context is still usable: re-zero the workspace and run normally
    dec.ws.zero_()
    dec.args.flags = 0
    out, _ = dec()
    dec.status()
    ref = oracle.decode_case(c)
    assert_attn_close(host_bits(out), ref["out"][:, 0])


# The pooled keys stream through a ring of 4 shared-memory stages of 256
# groups.  With 148 blocks, 1024 groups per block is 4 stages (the last in the
# last slot) and 1100 groups per block plus 9 is 5 stages with a partial last
# stage and a ragged last tile.
@pytest.mark.parametrize("groups", [148 * 1024, 148 * 1100 + 9])
def test_decode_stream_ring_stage_counts(groups):
    spec = synth.Spec(B=1, lengths=[4 * groups], H_i=8, k=512, H_q=16, plant_frac=0.05,
                      seed=208)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    got = run_decode(c, ref["k_pooled"], append=True, corrupt_last=True)
    assert np.array_equal(got["k_pooled"], ref["k_pooled"])
    check_against_oracle(c, got, ref)


def test_decode_append_repools_newest_group():
    spec = synth.Spec(B=3, lengths=[4096, 1024, 2000], H_i=8, k=128, H_q=32, seed=200)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    got = run_decode(c, ref["k_pooled"], append=True, corrupt_last=True)
    assert np.array_equal(got["k_pooled"], ref["k_pooled"])
    check_against_oracle(c, got, ref)


def test_decode_fewer_groups_than_k():
    spec = synth.Spec(B=2, lengths=[64, 8], L_cap=1024, H_i=4, k=64, H_q=16, seed=201)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    got = run_decode(c, ref["k_pooled"])
    assert (got["idx"][0, 16:] == -1).all() and (got["idx"][1, 2:] == -1).all()
    check_against_oracle(c, got, ref)


def test_decode_repeated_calls_reuse_workspace():
    spec = synth.Spec(B=2, lengths=[8192, 6000], H_i=8, k=256, H_q=64, seed=202)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    d = upload_case(c)
    dec = lcsw.Decoder(d["q_idx"][:, 0], d["w_head"][:, 0], dev_bf16(ref["k_pooled"]),
                       d["q"][:, 0], d["K"], d["V"], d["seq_len"], 4, c["k"], c["scale"])
    outs = [host_bits(dec()[0]).copy() for _ in range(3)]
    dec.status()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    assert_attn_close(outs[0], ref["out"][:, 0])


# ----------------------------------------------------------------- prefill --

def run_prefill(c, kp_cached, flags=0):
    d = upload_case(c)
    B, T, k = c["B"], c["T"], c["k"]
    kp = dev_bf16(kp_cached).clone()
    idx = torch.empty(B, T, k, dtype=torch.int32, device="cuda")
    out, lse = lcsw.prefill(d["q_idx"], d["w_head"], kp, d["k_idx"], d["pool_w"], d["q"], d["K"],
                            d["V"], d["seq_len"], c["P"], k, c["scale"], idx_out=idx, flags=flags)
    return dict(out=host_bits(out), lse=lse.cpu().numpy(), idx=idx.cpu().numpy(),
                k_pooled=host_bits(kp))


def _cached_part(kp_full, c):
    """Pooled cache as it stood before the chunk: the chunk's groups zeroed."""
    kp = kp_full.copy()
    for b in range(c["B"]):
        g0 = (int(c["seq_len"][b]) - c["T"]) // c["P"]
        kp[b, g0:] = 0
    return kp


@pytest.mark.parametrize("lengths,T,k", [([16384 + 256], 256, 512), ([3001, 2050], 48, 100)])
def test_prefill_reduced(lengths, T, k):
    spec = synth.Spec(B=len(lengths), lengths=lengths, T=T, prefill=True, H_i=8, k=k, H_q=32,
                      seed=210 + T)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    got = run_prefill(c, _cached_part(ref["k_pooled"], c))
    assert np.array_equal(got["k_pooled"], ref["k_pooled"])
    nd = selection_diff(got["idx"], ref["idx"], ref["scores"])
    assert nd == 0, f"{nd} rows differ by near-ties"
    assert_attn_close(got["out"], ref["out"])
    assert_lse_close(got["lse"], ref["lse"])


# T >= 64 with 8 indexer heads: the selection is fused with the tensor-core
# scoring (sample thresholds, candidates, exact top k from the candidates).
# The ragged case has a sequence shorter than k groups (every visible group
# selected) and group tiles past its end; the forced case sends every query
# through the dense-scores fallback.
@pytest.mark.parametrize("lengths,T,k,flags", [
    ([16384 + 256, 856], 256, 512, 0),
    ([16384 + 256], 256, 512, lcsw.PREFILL_FORCE_FALLBACK),
])
def test_prefill_fused_selection(lengths, T, k, flags):
    spec = synth.Spec(B=len(lengths), lengths=lengths, T=T, prefill=True, H_i=8, k=k, H_q=32,
                      seed=230 + len(lengths) + flags)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    got = run_prefill(c, _cached_part(ref["k_pooled"], c), flags=flags)
    nd = selection_diff(got["idx"], ref["idx"], ref["scores"])
    assert nd == 0, f"{nd} rows differ by near-ties"
    assert_attn_close(got["out"], ref["out"])
    assert_lse_close(got["lse"], ref["lse"])


# From 256 query rows the prefill attention runs on the tensor cores (chunks
# of 128 selected tokens, S and O accumulated in TMEM).  Edges: a sequence
# with fewer visible groups than k (padded selections), k*P not a multiple of
# 128 (a partial last chunk), 16 query heads (half of the head tile padded),
# P = 2, and rows of exactly three chunks (the last chunk's rescale is written
# after its vote, so the row-end fold must wait for a barrier).
@pytest.mark.parametrize("lengths,T,k,H_q,P", [([600, 5000], 128, 200, 16, 4),
                                               ([3000], 256, 70, 32, 2),
                                               ([4000], 256, 80, 32, 4)])
def test_prefill_tensor_core_attention_edges(lengths, T, k, H_q, P):
    spec = synth.Spec(B=len(lengths), lengths=lengths, T=T, prefill=True, H_i=8, k=k, H_q=H_q,
                      P=P, seed=250 + P)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    got = run_prefill(c, _cached_part(ref["k_pooled"], c))
    nd = selection_diff(got["idx"], ref["idx"], ref["scores"])
    assert nd == 0, f"{nd} rows differ by near-ties"
    assert_attn_close(got["out"], ref["out"])
    assert_lse_close(got["lse"], ref["lse"])


def test_prefill_tensor_core_attention_bounded_wait_reports_timeout():
    """The attention's first key chunk is never handed over: the MMA warp's
    bounded wait runs out, every role stops, the status reads TIMEOUT, and the
    next call on the same context is correct."""
    spec = synth.Spec(B=1, lengths=[3000], T=256, prefill=True, H_i=8, k=64, H_q=16, seed=260)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    kp = _cached_part(ref["k_pooled"], c)
    with pytest.raises(lcsw.LcswError) as ei:
        run_prefill(c, kp, flags=lcsw.PREFILL_TEST_SKIP_GATHER)
    assert ei.value.status == lcsw.ERR_TIMEOUT
    got = run_prefill(c, kp)
    assert_attn_close(got["out"], ref["out"])
    assert_lse_close(got["lse"], ref["lse"])


def test_prefill_fused_selection_exact_ties():
    # integer keys and queries with dyadic weights: exact scores with many equal
    # values, so the tie rule (lowest group first) decides many selections
    spec = synth.Spec(B=1, lengths=[8192 + 128], T=128, prefill=True, H_i=4, k=64, H_q=16,
                      idx_values="int3", w_mode="quarter_half", pool_mode="dyadic", seed=240)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    got = run_prefill(c, _cached_part(ref["k_pooled"], c))
    assert np.array_equal(got["idx"], ref["idx"])


@pytest.mark.parametrize("P,k", [(1, 2048), (2, 512), (8, 256)])
def test_decode_step_other_pool_sizes(P, k):
    """The persistent step with groups of 1 (the IndexPool-off ablation's
    k = 2048), 2 and 8 tokens, appending the newest group, over a ragged pair
    of sequences."""
    spec = synth.Spec(B=2, lengths=[96000 // P * P, 20000 // P * P], H_i=8, k=k, H_q=32, P=P,
                      plant_frac=0.05, seed=215 + P)
    c = synth.generate(spec)
    ref = oracle.decode_case(c)
    got = run_decode(c, ref["k_pooled"], append=True, corrupt_last=True)
    assert got["launches"] == 1
    assert np.array_equal(got["k_pooled"], ref["k_pooled"])
    check_against_oracle(c, got, ref)
