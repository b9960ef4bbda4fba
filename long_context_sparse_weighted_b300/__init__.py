"""Python binding of liblcsw.so: pooled-indexer sparse attention on B300.

Argument marshalling only.  Every step of the path runs in the library's CUDA
kernels; tensors are torch CUDA tensors (torch supplies device memory and the
current stream).  There is no CPU fallback: if liblcsw.so is missing or fails
to load, importing a function raises.

bf16 tensors may be torch.bfloat16 or int16/uint16 views of bf16 bits.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("LCSW_LIBRARY") or os.path.join(_HERE, "liblcsw.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "lcsw.h")

OK, ERR_INVALID_ARG, ERR_CUDA, ERR_UNSUPPORTED, ERR_TIMEOUT, ERR_WORKSPACE = range(6)

_lib = None

_vp, _i32, _i64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                              ctypes.c_size_t)


class DecodeArgs(ctypes.Structure):
    """Mirror of lcsw_decode_args."""
    _fields_ = [
        ("q_idx", _vp), ("w_head", _vp), ("k_pooled", _vp), ("sp_b", _i64),
        ("k_idx", _vp), ("sk_b", _i64), ("pool_w", _vp), ("sw_b", _i64),
        ("q", _vp), ("K", _vp), ("sK_b", _i64), ("V", _vp), ("sV_b", _i64),
        ("seq_len", _vp),
        ("B", _i32), ("G_max", _i32), ("H_i", _i32), ("d_idx", _i32), ("P", _i32), ("k", _i32),
        ("H_q", _i32), ("d_qk", _i32), ("d_v", _i32), ("scale", _f32),
        ("out", _vp), ("lse", _vp), ("idx_out", _vp), ("scores_out", _vp),
        ("flags", _i32),
    ]


FORCE_MULTIPASS_SELECT = 1
FORCE_MULTIKERNEL = 2
TEST_SKIP_ARRIVE = 4
PREFILL_FORCE_FALLBACK = 1  # lcsw_prefill_args.flags
PREFILL_TEST_SKIP_GATHER = 2


class PrefillArgs(ctypes.Structure):
    """Mirror of lcsw_prefill_args."""
    _fields_ = [
        ("q_idx", _vp), ("w_head", _vp), ("k_pooled", _vp), ("sp_b", _i64),
        ("k_idx", _vp), ("sk_b", _i64), ("pool_w", _vp), ("sw_b", _i64),
        ("q", _vp), ("K", _vp), ("sK_b", _i64), ("V", _vp), ("sV_b", _i64),
        ("seq_len", _vp),
        ("B", _i32), ("T", _i32), ("G_max", _i32), ("H_i", _i32), ("d_idx", _i32), ("P", _i32),
        ("k", _i32), ("H_q", _i32), ("d_qk", _i32), ("d_v", _i32), ("scale", _f32),
        ("out", _vp), ("lse", _vp), ("idx_out", _vp), ("flags", _i32),
    ]


_SIGNATURES = {
    "lcsw_last_error": ([], ctypes.c_char_p),
    "lcsw_version": ([], ctypes.c_char_p),
    "lcsw_pool_keys": ([_vp, _i64, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i64, _vp],
                       _i32),
    "lcsw_index_scores": ([_vp, _vp, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                           _vp, _vp], _i32),
    "lcsw_visible_counts": ([_vp, _vp, _i32, _i32, _i32, _vp, _vp], _i32),
    "lcsw_topk_workspace_size": ([_i64, _i32, _i32], _sz),
    "lcsw_topk_groups": ([_vp, _vp, _i64, _i32, _i32, _vp, _vp, _sz, _vp], _i32),
    "lcsw_sparse_attn_workspace_size": ([_i32, _i32, _i32, _i32, _i32, _i32], _sz),
    "lcsw_sparse_attn": ([_vp, _vp, _i64, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                          _i32, _i32, _f32, _vp, _vp, _vp, _sz, _vp], _i32),
    "lcsw_sparse_attn_noalloc": ([_vp, _vp, _i64, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32,
                                  _i32, _i32, _i32, _f32, _vp, _vp, _vp], _i32),
    "lcsw_decode_workspace_size": ([ctypes.POINTER(DecodeArgs)], _sz),
    "lcsw_decode_fused": ([ctypes.POINTER(DecodeArgs), _vp, _sz, _vp], _i32),
    "lcsw_decode_launches": ([ctypes.POINTER(DecodeArgs)], _i32),
    "lcsw_decode_reuse": ([ctypes.POINTER(DecodeArgs), _vp, _vp, _sz, _vp], _i32),
    "lcsw_quantize_keys_e4m3": ([_vp, _i64, _i32, _i32, _vp, _i64, _vp], _i32),
    "lcsw_decode_fused_e4m3": ([ctypes.POINTER(DecodeArgs), _vp, _i64, _vp, _sz, _vp], _i32),
    "lcsw_prefill_workspace_size": ([ctypes.POINTER(PrefillArgs)], _sz),
    "lcsw_prefill": ([ctypes.POINTER(PrefillArgs), _vp, _sz, _vp], _i32),
    "lcsw_quantize_rows_e4m3": ([_vp, _i64, _vp, _i32, _i32, _i32, _vp, _i64, _vp, _i64, _vp],
                                _i32),
    "lcsw_sparse_attn_kv8_workspace_size": ([_i32, _i32, _i32, _i32, _i32, _i32], _sz),
    "lcsw_sparse_attn_kv8": ([_vp, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i32,
                              _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _vp, _sz, _vp],
                             _i32),
    "lcsw_append_token": ([_vp, _i64, _vp, _i32, _vp, _i64, _i32, _vp, _i64, _i32, _vp, _i64,
                           _i32, _vp], _i32),
    "lcsw_quantize_rows_i8": ([_vp, _i64, _vp, _i32, _i32, _i32, _vp, _i64, _vp, _i64, _vp],
                              _i32),
    "lcsw_sparse_attn_kvi8": ([_vp, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i32,
                               _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _vp, _sz, _vp],
                              _i32),
    "lcsw_sparse_attn_mla_workspace_size": ([_i32, _i32, _i32, _i32, _i32], _sz),
    "lcsw_sparse_attn_mla": ([_vp, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _vp,
                              _vp, _vp, _sz, _vp], _i32),
    "lcsw_kda_step": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp], _i32),
    "lcsw_get_status": ([_vp, _vp], _i32),
    "lcsw_checks_enabled": ([], _i32),
    "lcsw_check_status": ([], _i32),
}


class LcswError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"lcsw status {status}: {msg}")
        self.status = status


def lib():
    """The loaded liblcsw.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; build it with "
                               "`python -m long_context_sparse_weighted_b300._build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(status: int):
    if status != OK:
        raise LcswError(status, lib().lcsw_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


_BF16_OK = (torch.bfloat16, torch.int16, torch.uint16)


def _bf16(t: torch.Tensor, name: str, ndim: int, inner_contig: bool = True):
    if t.dtype not in _BF16_OK:
        raise TypeError(f"{name} must be bf16 (or its 16-bit view), got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if inner_contig and t.shape[0] > 0 and not t[0].is_contiguous():
        raise ValueError(f"{name} must be contiguous apart from its batch stride")
    return t


def _dense(t: torch.Tensor, dtype, name: str):
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    return t


def version() -> str:
    return lib().lcsw_version().decode()


# --------------------------------------------------------------- primitives --

def pool_keys(k_idx, pool_w, seq_len, P, k_pooled, g_begin=None, g_span=None, stream=None):
    """IndexPool: k_pooled[b, g] = bf16(sum_j pool_w[b, g, j] * k_idx[b, P*g + j])."""
    _bf16(k_idx, "k_idx", 3)
    _bf16(k_pooled, "k_pooled", 3)
    if pool_w.dtype != torch.float32 or not pool_w[0].is_contiguous():
        raise ValueError("pool_w must be float32 [B][G][P], contiguous per sequence")
    _dense(seq_len, torch.int32, "seq_len")
    B, _, d = k_idx.shape
    if g_span is None:
        g_span = k_pooled.shape[1]
    _check(lib().lcsw_pool_keys(_ptr(k_idx), k_idx.stride(0), _ptr(pool_w), pool_w.stride(0),
                                _ptr(seq_len), _ptr(g_begin), B, int(g_span), d, P,
                                _ptr(k_pooled), k_pooled.stride(0), _stream(stream)))
    return k_pooled


def index_scores(q_idx, w_head, k_pooled, seq_len, P, G_max=None, q_pos=None, out=None,
                 stream=None):
    """Indexer scores [B][T][G_max] (fp32, -inf where not visible)."""
    _bf16(q_idx, "q_idx", 4)
    _bf16(k_pooled, "k_pooled", 3)
    _dense(w_head, torch.float32, "w_head")
    _dense(seq_len, torch.int32, "seq_len")
    B, T, H_i, d = q_idx.shape
    if G_max is None:
        G_max = k_pooled.shape[1]
    if out is None:
        out = torch.empty(B, T, G_max, dtype=torch.float32, device=q_idx.device)
    _check(lib().lcsw_index_scores(_ptr(q_idx), _ptr(w_head), _ptr(k_pooled),
                                   k_pooled.stride(0), _ptr(seq_len), _ptr(q_pos), B, T, H_i, d,
                                   P, int(G_max), _ptr(out), _stream(stream)))
    return out


def kda_step(qkv, conv_w, conv_state, g, beta, state, out=None, stream=None):
    """KDA step over T tokens: gated delta-rule recurrence after a causal short
    convolution (see lcsw_kda_step).  Updates `state` and `conv_state` in place
    and returns out [B][T][H][D] (bf16).

    qkv [B][T][3*H*D] bf16, conv_w [3*H*D][4] bf16, conv_state [B][3][3*H*D]
    bf16, g [B][T][H][D] fp32, beta [B][T][H] fp32, state [B][H][D][D] fp32.
    """
    _dense(qkv, torch.bfloat16, "qkv")
    _dense(conv_w, torch.bfloat16, "conv_w")
    _dense(conv_state, torch.bfloat16, "conv_state")
    _dense(g, torch.float32, "g")
    _dense(beta, torch.float32, "beta")
    _dense(state, torch.float32, "state")
    B, H, D, _ = state.shape
    T = qkv.shape[1]
    if qkv.shape != (B, T, 3 * H * D) or conv_w.shape != (3 * H * D, 4) or \
            conv_state.shape != (B, 3, 3 * H * D) or g.shape != (B, T, H, D) or \
            beta.shape != (B, T, H):
        raise ValueError("inconsistent KDA shapes")
    if out is None:
        out = torch.empty(B, T, H, D, dtype=torch.bfloat16, device=qkv.device)
    _dense(out, torch.bfloat16, "out")
    _check(lib().lcsw_kda_step(_ptr(qkv), _ptr(conv_w), _ptr(conv_state), _ptr(g), _ptr(beta),
                               _ptr(state), _ptr(out), B, T, H, D, _stream(stream)))
    return out


def visible_counts(seq_len, q_pos, B, T, P, stream=None):
    out = torch.empty(B, T, dtype=torch.int32, device=seq_len.device)
    _check(lib().lcsw_visible_counts(_ptr(seq_len), _ptr(q_pos), B, T, P, _ptr(out),
                                     _stream(stream)))
    return out


def topk_groups(scores, n_valid, k, out=None, ws=None, stream=None):
    """Top-k groups per row, ascending, -1 padded (rows = all leading dims).
    ws: optional uint8 workspace of lcsw_topk_workspace_size bytes (allocated
    here when missing; few long rows use it for the multi-block selection)."""
    _dense(scores, torch.float32, "scores")
    _dense(n_valid, torch.int32, "n_valid")
    G_max = scores.shape[-1]
    rows = scores.numel() // G_max if G_max else 0
    if out is None:
        out = torch.empty(*scores.shape[:-1], k, dtype=torch.int32, device=scores.device)
    nbytes = lib().lcsw_topk_workspace_size(rows, G_max, k)
    if ws is None and nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=scores.device)
    _check(lib().lcsw_topk_groups(_ptr(scores), _ptr(n_valid), rows, G_max, k, _ptr(out),
                                  _ptr(ws), nbytes, _stream(stream)))
    return out


def sparse_attn(q, K, V, seq_len, idx, P, scale, out=None, lse=None, ws=None, stream=None):
    """Attention of every query head over the tokens of the selected groups."""
    _bf16(q, "q", 4)
    _bf16(K, "K", 3)
    _bf16(V, "V", 3)
    _dense(idx, torch.int32, "idx")
    _dense(seq_len, torch.int32, "seq_len")
    B, T, H_q, d_qk = q.shape
    d_v = V.shape[2]
    k = idx.shape[-1]
    if out is None:
        out = torch.empty(B, T, H_q, d_v, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, T, H_q, dtype=torch.float32, device=q.device)
    nbytes = lib().lcsw_sparse_attn_workspace_size(B, T, H_q, d_v, k, P)
    if ws is None and nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check(lib().lcsw_sparse_attn(_ptr(q), _ptr(K), K.stride(0), _ptr(V), V.stride(0),
                                  _ptr(seq_len), _ptr(idx), B, T, H_q, d_qk, d_v, P, k,
                                  float(scale), _ptr(out), _ptr(lse), _ptr(ws), nbytes,
                                  _stream(stream)))
    return out, lse


def append_token(rows, seq_len, k_idx, K, V=None, stream=None):
    """Write each sequence's newest token (row seq_len[b] - 1) into k_idx, K
    and V from packed rows [B][d_idx + d_qk + d_v] (lcsw_append_token); V None
    for the MLA geometry (rows then hold d_idx + d_qk values)."""
    _bf16(rows, "rows", 2)
    _dense(seq_len, torch.int32, "seq_len")
    _bf16(k_idx, "k_idx", 3)
    _bf16(K, "K", 3)
    if V is not None:
        _bf16(V, "V", 3)
    B = rows.shape[0]
    d_v = V.shape[2] if V is not None else 0
    _check(lib().lcsw_append_token(_ptr(rows), rows.stride(0), _ptr(seq_len), B, _ptr(k_idx),
                                   k_idx.stride(0), k_idx.shape[2], _ptr(K), K.stride(0),
                                   K.shape[2], _ptr(V), V.stride(0) if V is not None else 0, d_v,
                                   _stream(stream)))


def _quantize_rows(fn, dtype, x, codes, scales, row_begin, n_rows, stream):
    _bf16(x, "x", 3)
    B, L, W = x.shape
    if codes is None:
        codes = torch.zeros(B, L, W, dtype=dtype, device=x.device)
    if scales is None:
        scales = torch.zeros(B, L, dtype=torch.float32, device=x.device)
    if n_rows is None:
        n_rows = L
    _check(fn(_ptr(x), x.stride(0), _ptr(row_begin), B, int(n_rows), W, _ptr(codes),
              codes.stride(0), _ptr(scales), scales.stride(0), _stream(stream)))
    return codes, scales


def quantize_rows_e4m3(x, codes=None, scales=None, row_begin=None, n_rows=None, stream=None):
    """bf16 cache x [B][L][width] -> E4M3 codes [B][L][width] (uint8) and one
    fp32 scale per row [B][L] (lcsw_quantize_rows_e4m3).  With row_begin [B]
    (int32) and n_rows, only rows [row_begin[b], row_begin[b] + n_rows) of
    each sequence are written."""
    return _quantize_rows(lib().lcsw_quantize_rows_e4m3, torch.uint8, x, codes, scales,
                          row_begin, n_rows, stream)


def quantize_rows_i8(x, codes=None, scales=None, row_begin=None, n_rows=None, stream=None):
    """bf16 cache x [B][L][width] -> INT8 codes [B][L][width] (int8) and one
    fp32 scale per row [B][L] (lcsw_quantize_rows_i8); the row window as in
    quantize_rows_e4m3."""
    return _quantize_rows(lib().lcsw_quantize_rows_i8, torch.int8, x, codes, scales, row_begin,
                          n_rows, stream)


def _quantized_kv_attn(fn, dtype, q, kc, ks, vc, vs, seq_len, idx, P, scale, out, lse, ws,
                       stream):
    _bf16(q, "q", 4)
    _dense(idx, torch.int32, "idx")
    _dense(seq_len, torch.int32, "seq_len")
    for t, n in ((kc, "kc"), (vc, "vc")):
        if t.dtype != dtype or not t.is_cuda or not t[0].is_contiguous():
            raise ValueError(f"{n} must be CUDA {dtype} [B][L][d], contiguous per sequence")
    B, T, H_q, d_qk = q.shape
    d_v = vc.shape[2]
    k = idx.shape[-1]
    if out is None:
        out = torch.empty(B, T, H_q, d_v, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, T, H_q, dtype=torch.float32, device=q.device)
    nbytes = lib().lcsw_sparse_attn_kv8_workspace_size(B, T, H_q, d_v, k, P)
    if ws is None and nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check(fn(_ptr(q), _ptr(kc), kc.stride(0), _ptr(ks), ks.stride(0), _ptr(vc), vc.stride(0),
              _ptr(vs), vs.stride(0), _ptr(seq_len), _ptr(idx), B, T, H_q, d_qk, d_v, P, k,
              float(scale), _ptr(out), _ptr(lse), _ptr(ws), nbytes, _stream(stream)))
    return out, lse


def sparse_attn_kv8(q, kc, ks, vc, vs, seq_len, idx, P, scale, out=None, lse=None, ws=None,
                    stream=None):
    """sparse_attn over an FP8 K/V cache (codes kc [B][L][d_qk], vc [B][L][d_v]
    uint8; one fp32 scale per token row ks, vs [B][L])."""
    return _quantized_kv_attn(lib().lcsw_sparse_attn_kv8, torch.uint8, q, kc, ks, vc, vs, seq_len,
                              idx, P, scale, out, lse, ws, stream)


def sparse_attn_kvi8(q, kc, ks, vc, vs, seq_len, idx, P, scale, out=None, lse=None, ws=None,
                     stream=None):
    """sparse_attn over an INT8 K/V cache (codes kc [B][L][d_qk], vc [B][L][d_v]
    int8; one fp32 scale per token row ks, vs [B][L])."""
    return _quantized_kv_attn(lib().lcsw_sparse_attn_kvi8, torch.int8, q, kc, ks, vc, vs, seq_len,
                              idx, P, scale, out, lse, ws, stream)


MLA_DQK, MLA_DV = 576, 512  # latent 512 + rotary 64; the latent is the value


def sparse_attn_mla(q, kv, seq_len, idx, P, scale, out=None, lse=None, ws=None, stream=None):
    """Attention in the MLA latent geometry: kv rows [c (512) | rope (64)] shared
    by every head, the latent c doubling as the value (lcsw_sparse_attn_mla).
    q [B][T][H_q][576], kv [B][L][576], idx [B][T][k] -> out [B][T][H_q][512]."""
    _bf16(q, "q", 4)
    _bf16(kv, "kv", 3)
    _dense(idx, torch.int32, "idx")
    _dense(seq_len, torch.int32, "seq_len")
    B, T, H_q, d_qk = q.shape
    if d_qk != MLA_DQK or kv.shape[2] != MLA_DQK:
        raise ValueError("MLA rows are 576 wide")
    k = idx.shape[-1]
    if out is None:
        out = torch.empty(B, T, H_q, MLA_DV, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, T, H_q, dtype=torch.float32, device=q.device)
    nbytes = lib().lcsw_sparse_attn_mla_workspace_size(B, T, H_q, k, P)
    if ws is None and nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check(lib().lcsw_sparse_attn_mla(_ptr(q), _ptr(kv), kv.stride(0), _ptr(seq_len), _ptr(idx),
                                      B, T, H_q, P, k, float(scale), _ptr(out), _ptr(lse),
                                      _ptr(ws), nbytes, _stream(stream)))
    return out, lse


def sparse_attn_noalloc(q, K, V, seq_len, idx, P, scale, out, lse=None, stream=None):
    """sparse_attn through the entry point that takes no workspace.

    The library keeps the split-K scratch in a fixed per-device array, so this
    call allocates nothing on the device: `out` (and `lse`, if wanted) are the
    caller's.  Calls that overlap in time on one device race on that scratch.
    """
    _bf16(q, "q", 4)
    _bf16(K, "K", 3)
    _bf16(V, "V", 3)
    _bf16(out, "out", 4)
    _dense(idx, torch.int32, "idx")
    _dense(seq_len, torch.int32, "seq_len")
    if lse is not None:
        _dense(lse, torch.float32, "lse")
    B, T, H_q, d_qk = q.shape
    d_v = V.shape[2]
    k = idx.shape[-1]
    _check(lib().lcsw_sparse_attn_noalloc(_ptr(q), _ptr(K), K.stride(0), _ptr(V), V.stride(0),
                                          _ptr(seq_len), _ptr(idx), B, T, H_q, d_qk, d_v, P, k,
                                          float(scale), _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


E4M3_TILE_BYTES = 1088  # 16 rows of 64 E4M3 codes, then their 16 fp32 scales


def e4m3_key_cache(B, G_max, device="cuda"):
    """An FP8 pooled-key cache of B sequences x ceil(G_max/16) tiles (uint8)."""
    return torch.zeros(B, (G_max + 15) // 16 * E4M3_TILE_BYTES, dtype=torch.uint8, device=device)


def quantize_keys_e4m3(k_pooled, kq, n_groups=None, stream=None):
    """Groups [0, n_groups) of every sequence's bf16 pooled keys into the FP8
    cache kq ([B][tiles * 1088] uint8): per-row scale amax/448, E4M3 codes."""
    _bf16(k_pooled, "k_pooled", 3)
    if kq.dtype != torch.uint8 or not kq.is_cuda or not kq[0].is_contiguous():
        raise ValueError("kq must be a CUDA uint8 tensor [B][bytes]")
    B = k_pooled.shape[0]
    n = k_pooled.shape[1] if n_groups is None else int(n_groups)
    _check(lib().lcsw_quantize_keys_e4m3(_ptr(k_pooled), k_pooled.stride(0), B, n, _ptr(kq),
                                         kq.stride(0), _stream(stream)))
    return kq


# ------------------------------------------------------------ decode step ---

class Decoder:
    """One decode step of the whole path through lcsw_decode_fused.

    Holds the argument struct and a zero-initialised workspace; tensors are
    bound once and may be refilled in place between calls.
    """

    def __init__(self, q_idx, w_head, k_pooled, q, K, V, seq_len, P, k, scale,
                 k_idx=None, pool_w=None, out=None, lse=None, idx_out=None, scores_out=None,
                 G_max=None, flags=0, kq=None):
        """kq: an FP8 pooled-key cache (e4m3_key_cache) to score from instead of
        the bf16 k_pooled (lcsw_decode_fused_e4m3); k_pooled may then be None
        when G_max is given."""
        _bf16(q_idx, "q_idx", 3)
        if kq is None or k_pooled is not None:
            _bf16(k_pooled, "k_pooled", 3)
        _bf16(q, "q", 3)
        _bf16(K, "K", 3)
        if V is not None:
            _bf16(V, "V", 3)
        _dense(w_head, torch.float32, "w_head")
        _dense(seq_len, torch.int32, "seq_len")
        B, H_i, d_idx = q_idx.shape
        H_q, d_qk = q.shape[1], q.shape[2]
        # V None: the MLA latent geometry (576-wide K rows whose latent is the value)
        d_v = V.shape[2] if V is not None else MLA_DV
        dev = q.device
        self.out = out if out is not None else torch.empty(B, H_q, d_v, dtype=torch.bfloat16,
                                                           device=dev)
        self.lse = lse if lse is not None else torch.empty(B, H_q, dtype=torch.float32,
                                                           device=dev)
        self.idx_out, self.scores_out = idx_out, scores_out
        self._keep = (q_idx, w_head, k_pooled, q, K, V, seq_len, k_idx, pool_w)
        a = DecodeArgs()
        a.q_idx, a.w_head = q_idx.data_ptr(), w_head.data_ptr()
        if k_pooled is not None:
            a.k_pooled, a.sp_b = k_pooled.data_ptr(), k_pooled.stride(0)
        if k_idx is not None:
            _bf16(k_idx, "k_idx", 3)
            a.k_idx, a.sk_b = k_idx.data_ptr(), k_idx.stride(0)
            a.pool_w, a.sw_b = pool_w.data_ptr(), pool_w.stride(0)
        a.q = q.data_ptr()
        a.K, a.sK_b = K.data_ptr(), K.stride(0)
        if V is not None:
            a.V, a.sV_b = V.data_ptr(), V.stride(0)
        a.seq_len = seq_len.data_ptr()
        a.B, a.G_max = B, int(G_max if G_max is not None else k_pooled.shape[1])
        self.kq = kq
        if kq is not None and (kq.dtype != torch.uint8 or not kq.is_cuda):
            raise ValueError("kq must be a CUDA uint8 tensor")
        a.H_i, a.d_idx, a.P, a.k = H_i, d_idx, P, k
        a.H_q, a.d_qk, a.d_v, a.scale = H_q, d_qk, d_v, float(scale)
        a.out, a.lse = self.out.data_ptr(), self.lse.data_ptr()
        a.idx_out = idx_out.data_ptr() if idx_out is not None else None
        a.scores_out = scores_out.data_ptr() if scores_out is not None else None
        a.flags = int(flags)
        self.args = a
        self.ws_bytes = lib().lcsw_decode_workspace_size(ctypes.byref(a))
        # the FP8 step is always the one persistent launch (or an error)
        self.launches_per_call = 1 if kq is not None else \
            lib().lcsw_decode_launches(ctypes.byref(a))
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)

    def rebind(self, **tensors):
        """Point the step at other tensors of identical shape (e.g. rotated caches)."""
        a = self.args
        for name, t in tensors.items():
            setattr(a, name, t.data_ptr())
        self._rebound = tensors

    def __call__(self, stream=None):
        if self.kq is not None:
            _check(lib().lcsw_decode_fused_e4m3(ctypes.byref(self.args), _ptr(self.kq),
                                                self.kq.stride(0),
                                                ctypes.c_void_p(self.ws.data_ptr()),
                                                self.ws_bytes, _stream(stream)))
        else:
            _check(lib().lcsw_decode_fused(ctypes.byref(self.args),
                                           ctypes.c_void_p(self.ws.data_ptr()), self.ws_bytes,
                                           _stream(stream)))
        return self.out, self.lse

    def status(self, stream=None):
        _check(lib().lcsw_get_status(ctypes.c_void_p(self.ws.data_ptr()), _stream(stream)))


class ReuseStep:
    """A DSA layer's decode step that reuses another layer's selection
    (lcsw_decode_reuse): attention of q over the groups idx_in[b][0..k),
    with no indexer scores or top-k of its own."""

    def __init__(self, q, K, V, seq_len, idx_in, P, scale, out=None, lse=None, ws=None, flags=0):
        _bf16(q, "q", 3)
        _bf16(K, "K", 3)
        if V is not None:
            _bf16(V, "V", 3)
        _dense(seq_len, torch.int32, "seq_len")
        _dense(idx_in, torch.int32, "idx_in")
        B, H_q, d_qk = q.shape
        d_v = V.shape[2] if V is not None else MLA_DV
        k = idx_in.shape[-1]
        dev = q.device
        self.out = out if out is not None else torch.empty(B, H_q, d_v, dtype=torch.bfloat16,
                                                           device=dev)
        self.lse = lse if lse is not None else torch.empty(B, H_q, dtype=torch.float32,
                                                           device=dev)
        self._keep = (q, K, V, seq_len, idx_in)
        a = DecodeArgs()
        a.q = q.data_ptr()
        a.K, a.sK_b = K.data_ptr(), K.stride(0)
        if V is not None:
            a.V, a.sV_b = V.data_ptr(), V.stride(0)
        a.seq_len = seq_len.data_ptr()
        a.B, a.G_max, a.H_i, a.d_idx, a.P, a.k = B, 0, 1, 64, P, k
        a.H_q, a.d_qk, a.d_v, a.scale = H_q, d_qk, d_v, float(scale)
        a.out, a.lse = self.out.data_ptr(), self.lse.data_ptr()
        a.flags = int(flags)
        self.args = a
        self.idx_in = idx_in
        self.ws_bytes = lib().lcsw_decode_workspace_size(ctypes.byref(a))
        # a decode workspace is zero-filled before its first use (a shared one,
        # e.g. the selecting layer's, is already in that state between calls)
        self.ws = ws if ws is not None else torch.zeros(self.ws_bytes, dtype=torch.uint8,
                                                        device=dev)

    def __call__(self, stream=None):
        _check(lib().lcsw_decode_reuse(ctypes.byref(self.args), ctypes.c_void_p(self.idx_in.data_ptr()),
                                       ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(),
                                       _stream(stream)))
        return self.out, self.lse

    def status(self, stream=None):
        """Raise if a bounded device wait of an earlier call ran out (synchronises)."""
        _check(lib().lcsw_get_status(ctypes.c_void_p(self.ws.data_ptr()), _stream(stream)))


def decode_fused(q_idx, w_head, k_pooled, q, K, V, seq_len, P, k, scale, **kw):
    """One-shot decode step; returns (out, lse, decoder)."""
    d = Decoder(q_idx, w_head, k_pooled, q, K, V, seq_len, P, k, scale, **kw)
    out, lse = d()
    return out, lse, d


def prefill(q_idx, w_head, k_pooled, k_idx, pool_w, q, K, V, seq_len, P, k, scale,
            out=None, lse=None, idx_out=None, G_max=None, flags=0, stream=None, ws=None,
            check=True):
    """Chunked prefill of T query tokens per sequence (the last T of each cache).

    ws: optional uint8 device workspace of at least lcsw_prefill_workspace_size
    bytes whose first 256 bytes (the status word) are zero; reused across
    calls it needs no clearing, since a status check clears the word.
    check: read the status word after the call (synchronises the stream)."""
    _bf16(q_idx, "q_idx", 4)
    _bf16(q, "q", 4)
    B, T, H_i, d_idx = q_idx.shape
    H_q, d_qk = q.shape[2], q.shape[3]
    d_v = V.shape[2]
    dev = q.device
    if out is None:
        out = torch.empty(B, T, H_q, d_v, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(B, T, H_q, dtype=torch.float32, device=dev)
    a = PrefillArgs()
    a.q_idx, a.w_head = q_idx.data_ptr(), w_head.data_ptr()
    a.k_pooled, a.sp_b = k_pooled.data_ptr(), k_pooled.stride(0)
    a.k_idx, a.sk_b = k_idx.data_ptr(), k_idx.stride(0)
    a.pool_w, a.sw_b = pool_w.data_ptr(), pool_w.stride(0)
    a.q = q.data_ptr()
    a.K, a.sK_b = K.data_ptr(), K.stride(0)
    a.V, a.sV_b = V.data_ptr(), V.stride(0)
    a.seq_len = seq_len.data_ptr()
    a.B, a.T = B, T
    a.G_max = int(G_max if G_max is not None else k_pooled.shape[1])
    a.H_i, a.d_idx, a.P, a.k = H_i, d_idx, P, k
    a.H_q, a.d_qk, a.d_v, a.scale = H_q, d_qk, d_v, float(scale)
    a.out, a.lse = out.data_ptr(), lse.data_ptr()
    a.idx_out = idx_out.data_ptr() if idx_out is not None else None
    a.flags = int(flags)
    nbytes = lib().lcsw_prefill_workspace_size(ctypes.byref(a))
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        ws[:256].zero_()  # the status word; every other region is written before it is read
    elif ws.numel() < nbytes:
        raise ValueError(f"prefill workspace too small: {ws.numel()} < {nbytes} bytes")
    _check(lib().lcsw_prefill(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                              _stream(stream)))
    if check:
        _check(lib().lcsw_get_status(ctypes.c_void_p(ws.data_ptr()), _stream(stream)))
    return out, lse
