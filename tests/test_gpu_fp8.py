"""FP8 (E4M3) pooled indexer keys on the GPU against the oracle's FP8 leg.

lcsw_quantize_keys_e4m3 must give the oracle's codes and scales bit for bit;
lcsw_decode_fused_e4m3 must score like the oracle's FP8 indexer (exactly on
inputs whose products and sums are exact in fp32, within the score tolerance
otherwise), select the same groups and attend over them.  The tile-major
cache layout (16 rows of 64 codes, then 16 fp32 scales) is packed here from
the oracle's row-major codes, so the decode tests do not depend on the GPU
quantizer.
"""
import numpy as np
import pytest
import torch

import long_context_sparse_weighted_b300 as lcsw
import oracle
import synth
from gpu_util import (assert_attn_close, assert_lse_close, assert_scores_close, dev, dev_bf16,
                      host_bits, selection_diff, upload_case)

pytestmark = pytest.mark.gpu
TILE = lcsw.E4M3_TILE_BYTES


def pack_tiles(codes, scales):
    """Row-major codes [B][G][64] and scales [B][G] -> the tile-major cache."""
    B, G, _ = codes.shape
    tiles = (G + 15) // 16
    out = np.zeros((B, tiles, TILE), np.uint8)
    cp = np.zeros((B, tiles * 16, 64), np.uint8)
    sp = np.zeros((B, tiles * 16), np.float32)
    cp[:, :G] = codes
    sp[:, :G] = scales
    out[:, :, :1024] = cp.reshape(B, tiles, 1024)
    out[:, :, 1024:] = sp.reshape(B, tiles, 16).view(np.uint8).reshape(B, tiles, 64)
    return out.reshape(B, tiles * TILE)


def unpack_tiles(kq, G):
    B = kq.shape[0]
    t = kq.reshape(B, -1, TILE)
    codes = t[:, :, :1024].reshape(B, -1, 64)[:, :G]
    scales = np.ascontiguousarray(t[:, :, 1024:]).view(np.float32).reshape(B, -1)[:, :G]
    return codes, scales


def test_quantize_keys_bit_exact():
    rng = np.random.default_rng(70)
    B, G = 3, 700
    x = rng.standard_normal((B, G, 64)).astype(np.float32)
    x[0, 0] = 0.0                                     # all-zero row: scale 0, codes 0
    x[0, 1] = 0.0
    x[0, 1, 5] = -0.0                                 # signed zero beside a real value
    x[0, 1, 7] = 3.0
    x[1, 2] *= 1e-30                                  # subnormal quotients
    x[1, 3] *= 1e30                                   # large magnitudes
    x[1, 6] *= 1e-37                                  # a scale whose reciprocal overflows
    x[2, 4, :] = np.linspace(-448.0, 448.0, 64)        # amax 448: scale 1, E4M3 grid
    x[2, 5, :] = np.arange(64) * 0.5 + 1.0             # many midpoints between codes
    kp = (x.view(np.uint32) >> 16).astype(np.uint16)
    kp[0, 1, 5] = 0x8000
    codes, scales = oracle.quantize_rows_e4m3(kp)
    kq = lcsw.e4m3_key_cache(B, G)
    lcsw.quantize_keys_e4m3(dev_bf16(kp), kq)
    got_c, got_s = unpack_tiles(kq.cpu().numpy(), G)
    assert np.array_equal(got_s.view(np.uint32), scales.view(np.uint32))
    bad = np.argwhere(got_c != codes)
    assert bad.size == 0, f"{len(bad)} codes differ, e.g. {bad[:4].tolist()}"


def _fp8_oracle(c, kp):
    """The oracle's FP8 retrieval step: quantized keys and queries, FP8 scores,
    top-k, attention."""
    ck, sk = oracle.quantize_rows_e4m3(kp)
    cq, sq = oracle.quantize_rows_e4m3(c["q_idx"])
    s = oracle.index_scores_e4m3(cq, sq, c["w_head"], ck, sk, c["seq_len"], c["P"])
    nv = oracle.visible_counts(c["seq_len"], None, c["B"], 1, c["P"])
    idx = oracle.topk(s, nv, c["k"])
    out, lse = oracle.sparse_attn(c["q"], c["K"], c["V"], c["seq_len"], idx, c["P"], c["scale"])
    return dict(scores=s, idx=idx, out=out, lse=lse, ck=ck, sk=sk)


def _run_fp8(c, kq_host, append=False):
    d = upload_case(c)
    B, k = c["B"], c["k"]
    G_max = c["G_max"]
    kq = dev(kq_host)
    idx = torch.empty(B, k, dtype=torch.int32, device="cuda")
    scores = torch.empty(B, G_max, dtype=torch.float32, device="cuda")
    kw = dict(idx_out=idx, scores_out=scores, kq=kq, G_max=G_max)
    if append:
        kw.update(k_idx=d["k_idx"], pool_w=d["pool_w"])
    dec = lcsw.Decoder(d["q_idx"][:, 0], d["w_head"][:, 0], None, d["q"][:, 0], d["K"], d["V"],
                       d["seq_len"], c["P"], k, c["scale"], **kw)
    assert dec.launches_per_call == 1
    out, lse = dec()
    dec.status()
    return dict(out=host_bits(out), lse=lse.cpu().numpy(), idx=idx.cpu().numpy(),
                scores=scores.cpu().numpy(), kq=kq.cpu().numpy())


def test_fp8_decode_exact_on_representable_inputs():
    # keys and queries drawn from {-2, -1, 0, 1, 2} with one +-448 per row:
    # every scale is 1, every code exact, every dot product an integer below
    # 2^24, and head weights in {1/4, 1/2}: fp32 scores are exact
    spec = synth.Spec(B=2, lengths=[8192, 6000], H_i=8, k=128, H_q=32, seed=71,
                      w_mode="quarter_half")
    c = synth.generate(spec)
    rng = np.random.default_rng(71)
    B, G = spec.B, c["G_max"]
    kv = rng.integers(-2, 3, (B, G, 64)).astype(np.float32)
    kv[:, :, 0] = 448.0 * rng.choice([-1.0, 1.0], (B, G))
    qv = rng.integers(-2, 3, c["q_idx"].shape).astype(np.float32)
    qv[..., 0] = 448.0
    kp = (kv.view(np.uint32) >> 16).astype(np.uint16)
    c["q_idx"] = (qv.view(np.uint32) >> 16).astype(np.uint16)
    ref = _fp8_oracle(c, kp)
    got = _run_fp8(c, pack_tiles(ref["ck"], ref["sk"]))
    assert np.array_equal(got["scores"], ref["scores"][:, 0])
    assert np.array_equal(got["idx"], ref["idx"][:, 0])
    assert_attn_close(got["out"], ref["out"][:, 0])
    assert_lse_close(got["lse"], ref["lse"][:, 0])


@pytest.mark.parametrize("name,factor", [("decode_1m", 16), ("decode_b8", 16),
                                         ("ragged_b64", 32)])
def test_fp8_decode_matches_the_fp8_oracle(name, factor):
    spec = synth.shrink(synth.named(name), factor)
    c = synth.generate(spec)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], c["P"])
    ref = _fp8_oracle(c, kp)
    got = _run_fp8(c, pack_tiles(ref["ck"], ref["sk"]))
    assert_scores_close(got["scores"], ref["scores"][:, 0])
    nd = selection_diff(got["idx"], ref["idx"][:, 0], ref["scores"][:, 0])
    assert nd == 0, f"{nd} rows selected a different (near-tie) set"
    assert_attn_close(got["out"], ref["out"][:, 0])
    assert_lse_close(got["lse"], ref["lse"][:, 0])


def test_fp8_decode_append_quantizes_the_newest_group():
    spec = synth.Spec(B=3, lengths=[40000, 9000, 123456 // 4 * 4], H_i=8, k=512, H_q=64,
                      plant_frac=0.05, seed=72)
    c = synth.generate(spec)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], c["P"])
    ref = _fp8_oracle(c, kp)
    ck, sk = ref["ck"].copy(), ref["sk"].copy()
    for b in range(spec.B):  # a stale newest group in the cache: the step re-pools it
        g = int(c["seq_len"][b]) // 4 - 1
        ck[b, g] = 0x38
        sk[b, g] = 7.0
    got = _run_fp8(c, pack_tiles(ck, sk), append=True)
    codes, scales = unpack_tiles(got["kq"], c["G_max"])
    assert np.array_equal(codes, ref["ck"])
    assert np.array_equal(scales.view(np.uint32), ref["sk"].view(np.uint32))
    assert_scores_close(got["scores"], ref["scores"][:, 0])
    assert selection_diff(got["idx"], ref["idx"][:, 0], ref["scores"][:, 0]) == 0
    assert_attn_close(got["out"], ref["out"][:, 0])


@pytest.mark.slow
def test_fp8_decode_full_size_decode_1m():
    """The benchmarked FP8-keys step: decode_1m's 262,144 groups quantized on
    the device, the newest group re-pooled and quantized by the step, against
    the oracle's FP8 step (its own quantizer, scores, top-k, attention)."""
    spec = synth.named("decode_1m")
    c = synth.generate(spec)
    kp = oracle.pool_keys(c["k_idx"], c["pool_w"], c["seq_len"], c["P"])
    ref = _fp8_oracle(c, kp)
    got = _run_fp8(c, pack_tiles(ref["ck"], ref["sk"]), append=True)
    codes, scales = unpack_tiles(got["kq"], c["G_max"])
    assert np.array_equal(codes, ref["ck"])
    assert np.array_equal(scales.view(np.uint32), ref["sk"].view(np.uint32))
    assert_scores_close(got["scores"], ref["scores"][:, 0])
    assert selection_diff(got["idx"], ref["idx"][:, 0], ref["scores"][:, 0]) == 0
    assert_attn_close(got["out"], ref["out"][:, 0])
    assert_lse_close(got["lse"], ref["lse"][:, 0])
