"""Helpers shared by the GPU parity tests: upload, tolerance checks.

Tolerances, and the arithmetic they come from:
  pooled keys, selected indices, visible counts   bit-exact (correctly rounded
                   bf16 of the exact pooled sum; integer work)
  indexer scores   |s_gpu - s_ref| <= 1e-5 * max(1, max_g |s_ref|)  per row
                   (fp32 accumulation of 64 exact bf16 products against fp64)
  attention out    max |o_gpu - o_ref| <= 2e-2 and
                   ||o_gpu - o_ref||_2 / ||o_ref||_2 <= 1e-2          per (b, t) row
                   (bf16 probabilities in the value product, fp32 sums,
                   bf16 output)
  lse              |lse_gpu - lse_ref| <= 1e-3 + 1e-4 |lse_ref|  (fp32 sums)
"""
import numpy as np
import torch

import synth

SCORE_RTOL = 1e-5
ATTN_MAX_ABS = 2e-2
ATTN_REL_L2 = 1e-2


def dev_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def upload_case(c: dict, device="cuda") -> dict:
    d = dict(seq_len=dev(c["seq_len"]), k_idx=dev_bf16(c["k_idx"]), pool_w=dev(c["pool_w"]),
             q_idx=dev_bf16(c["q_idx"]), w_head=dev(c["w_head"]), q=dev_bf16(c["q"]))
    if c.get("q_pos") is not None:
        d["q_pos"] = dev(c["q_pos"])
    if "K" in c:
        d["K"] = dev_bf16(c["K"])
        d["V"] = dev_bf16(c["V"])
    return d


def assert_scores_close(got: np.ndarray, ref: np.ndarray, rtol=SCORE_RTOL):
    got = got.reshape(-1, got.shape[-1])
    ref = ref.reshape(-1, ref.shape[-1])
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), "visibility mask differs"
    assert (got[~fin] == ref[~fin]).all()
    scale = np.maximum(1.0, np.abs(np.where(fin, ref, 0.0)).max(axis=1, keepdims=True))
    err = np.abs(np.where(fin, got, 0.0).astype(np.float64) - np.where(fin, ref, 0.0))
    worst = (err / scale).max()
    assert worst <= rtol, f"score error {worst:.3g} x row scale > {rtol}"
    return worst


def assert_attn_close(got_bits: np.ndarray, ref_bits: np.ndarray):
    g = synth.bf16_to_f32(got_bits).astype(np.float64)
    r = synth.bf16_to_f32(ref_bits).astype(np.float64)
    rows = g.shape[0] * g.shape[1] if g.ndim == 4 else g.shape[0]
    g = g.reshape(rows, -1)
    r = r.reshape(rows, -1)
    assert np.isfinite(g).all()
    max_abs = np.abs(g - r).max()
    rel = np.linalg.norm(g - r, axis=1) / np.maximum(np.linalg.norm(r, axis=1), 1e-30)
    assert max_abs <= ATTN_MAX_ABS, f"max abs error {max_abs:.3g}"
    assert rel.max() <= ATTN_REL_L2, f"relative L2 error {rel.max():.3g}"
    return max_abs, rel.max()


def assert_lse_close(got: np.ndarray, ref: np.ndarray):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert (got[~fin] == ref[~fin]).all()
    err = np.abs(got[fin].astype(np.float64) - ref[fin])
    assert (err <= 1e-3 + 1e-4 * np.abs(ref[fin])).all(), f"lse error {err.max():.3g}"


def selection_diff(idx_gpu: np.ndarray, idx_ref: np.ndarray, scores_ref: np.ndarray,
                   rtol=SCORE_RTOL):
    """Rows whose selections differ, checking each difference is a near-tie.

    idx_*: [rows][k] (ascending, -1 padded); scores_ref: [rows][G] (oracle).
    A group may be swapped only if its oracle score lies within the score
    tolerance of the row's k-th oracle score.  Returns the number of rows that
    differ (each verified to be a near-tie swap).
    """
    idx_gpu = idx_gpu.reshape(-1, idx_gpu.shape[-1])
    idx_ref = idx_ref.reshape(-1, idx_ref.shape[-1])
    scores_ref = scores_ref.reshape(-1, scores_ref.shape[-1])
    nd = 0
    for r in range(idx_gpu.shape[0]):
        a, b = idx_gpu[r], idx_ref[r]
        assert (np.diff(a[a >= 0]) > 0).all(), "GPU selection not strictly ascending"
        assert (a < 0).sum() == (b < 0).sum(), "different number of selected groups"
        if np.array_equal(a, b):
            continue
        nd += 1
        s = scores_ref[r]
        fin = np.isfinite(s)
        scale = max(1.0, np.abs(s[fin]).max())
        kth = s[b[b >= 0]].min()
        for g in set(a[a >= 0]) ^ set(b[b >= 0]):
            assert abs(float(s[g]) - float(kth)) <= 2 * rtol * scale, (
                f"row {r}: group {g} score {s[g]} not within tolerance of k-th {kth}")
    return nd
