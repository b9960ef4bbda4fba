"""CPU oracle of the pooled-indexer sparse-attention path (ctypes over oracle.c).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  The CUDA library never
imports, links or calls it, and it shares no code with the library.

Every function takes and returns numpy arrays; bf16 tensors are uint16 bit
patterns.  Arithmetic is fp64 (see oracle.c for the step-by-step definition
and the passages of the release notes each step follows).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _declare(lib):
    P, I32, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_bf16_from_double.argtypes = [D]
    lib.oracle_bf16_from_double.restype = ctypes.c_uint16
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = D
    lib.oracle_e4m3_from_double.argtypes = [D]
    lib.oracle_e4m3_from_double.restype = ctypes.c_uint8
    lib.oracle_quantize_rows_e4m3.argtypes = [P, I64, I32, P, P]
    lib.oracle_index_scores_e4m3.argtypes = [P, P, P, P, P, I64, P, P, I32, I32, I32, I32, I32,
                                             I64, P]
    lib.oracle_sparse_attn_e4m3kv.argtypes = [P, P, I64, P, I64, P, I64, P, I64, P, P, I32, I32,
                                              I32, I32, I32, I32, I32, D, P, P]
    lib.oracle_sparse_attn_e4m3kv.restype = None
    lib.oracle_i8_value.argtypes = [ctypes.c_int8, ctypes.c_float]
    lib.oracle_i8_value.restype = D
    lib.oracle_i8_from_double.argtypes = [D, ctypes.c_float]
    lib.oracle_i8_from_double.restype = ctypes.c_int8
    lib.oracle_quantize_rows_i8.argtypes = [P, I64, I32, P, P]
    lib.oracle_quantize_rows_i8.restype = None
    lib.oracle_sparse_attn_i8kv.argtypes = [P, P, I64, P, I64, P, I64, P, I64, P, P, I32, I32,
                                            I32, I32, I32, I32, I32, D, P, P]
    lib.oracle_sparse_attn_i8kv.restype = None
    lib.oracle_pool_keys.argtypes = [P, I64, P, I64, P, I32, I32, I32, P, I64]
    lib.oracle_visible_counts.argtypes = [P, P, I32, I32, I32, P]
    lib.oracle_index_scores.argtypes = [P, P, P, I64, P, P, I32, I32, I32, I32, I32, I64, P]
    lib.oracle_topk.argtypes = [P, P, I64, I64, I32, P]
    lib.oracle_sparse_attn.argtypes = [P, P, I64, P, I64, P, P, I32, I32, I32, I32, I32,
                                       I32, I32, D, P, P]
    lib.oracle_retrieval_step.argtypes = [P, P, P, I64, P, P, I64, P, I64, P, P, I32, I32,
                                          I32, I32, I32, I64, I32, I32, I32, I32, D, P, P,
                                          P, P]
    for f in ("oracle_pool_keys", "oracle_visible_counts", "oracle_index_scores",
              "oracle_topk", "oracle_sparse_attn", "oracle_retrieval_step"):
        getattr(lib, f).restype = None
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def compile_variant(src_text: str, so_path: str) -> None:
    """Compile a (deliberately altered) copy of oracle.c for mutation tests."""
    c_path = so_path[:-3] + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", *_CFLAGS, "-o", so_path, c_path, "-lm"])


class use_library:
    """Context manager: route this module's functions to another oracle build."""

    def __init__(self, so_path: str):
        self.path = so_path

    def __enter__(self):
        global _lib
        self.saved = _lib
        _lib = _declare(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.asarray(a)
    assert a.dtype == np.dtype(dtype), (a.dtype, dtype)
    return np.ascontiguousarray(a)


def bf16_from_double(x: float) -> int:
    return int(_load().oracle_bf16_from_double(float(x)))


def pool_keys(k_idx, pool_w, seq_len, P, out=None):
    """kbar[b,g,:] = bf16(sum_j alpha[b,g,j] * k[b,P*g+j,:]) for g < seq_len[b]//P."""
    k_idx = _c(k_idx, np.uint16)
    pool_w = _c(pool_w, np.float32)
    seq_len = _c(seq_len, np.int32)
    B, L_max, d = k_idx.shape
    G_max = pool_w.shape[1]
    assert pool_w.shape == (B, G_max, P)
    if out is None:
        out = np.zeros((B, G_max, d), np.uint16)
    _load().oracle_pool_keys(_p(k_idx), L_max * d, _p(pool_w), G_max * P, _p(seq_len), B, d, P,
                             _p(out), out.shape[1] * d)
    return out


def visible_counts(seq_len, q_pos, B, T, P):
    seq_len = _c(seq_len, np.int32)
    qp = None if q_pos is None else _c(q_pos, np.int32)
    out = np.zeros((B, T), np.int32)
    _load().oracle_visible_counts(_p(seq_len), _p(qp), B, T, P, _p(out))
    return out


def index_scores(q_idx, w_head, k_pooled, seq_len, P, q_pos=None):
    """s[b,t,g] = sum_h w[b,t,h] * relu(q[b,t,h,:] . kbar[b,g,:]); -inf if not visible."""
    q_idx = _c(q_idx, np.uint16)
    w_head = _c(w_head, np.float32)
    k_pooled = _c(k_pooled, np.uint16)
    seq_len = _c(seq_len, np.int32)
    B, T, H_i, d = q_idx.shape
    G_max = k_pooled.shape[1]
    qp = None if q_pos is None else _c(q_pos, np.int32)
    out = np.empty((B, T, G_max), np.float32)
    _load().oracle_index_scores(_p(q_idx), _p(w_head), _p(k_pooled), G_max * d, _p(seq_len),
                                _p(qp), B, T, H_i, d, P, G_max, _p(out))
    return out


def e4m3_value(code: int) -> float:
    """Value of an e4m3 code (OCP FP8 E4M3; NaN for S.1111.111)."""
    return _load().oracle_e4m3_value(int(code))


def e4m3_from_double(x: float) -> int:
    """Nearest e4m3 code, ties to the even code, saturating at +-448."""
    return int(_load().oracle_e4m3_from_double(float(x)))


def quantize_rows_e4m3(x):
    """bf16 rows [..., d] -> (e4m3 codes [..., d] uint8, fp32 scale per row = amax/448)."""
    x = _c(x, np.uint16)
    d = x.shape[-1]
    rows = int(np.prod(x.shape[:-1]))
    code = np.empty(x.shape, np.uint8)
    scale = np.empty(x.shape[:-1], np.float32)
    _load().oracle_quantize_rows_e4m3(_p(x), rows, d, _p(code), _p(scale))
    return code, scale


def sparse_attn_e4m3kv(q, kc, ks, vc, vs, seq_len, idx, P, scale):
    """Attention over an FP8 K/V cache: element = e4m3(code) * the token row's
    scale.  kc [B][L][d_qk], vc [B][L][d_v] uint8 codes; ks, vs [B][L] fp32."""
    q = _c(q, np.uint16)
    kc, vc = _c(kc, np.uint8), _c(vc, np.uint8)
    ks, vs = _c(ks, np.float32), _c(vs, np.float32)
    seq_len = _c(seq_len, np.int32)
    idx = _c(idx, np.int32)
    B, T, H_q, d_qk = q.shape
    d_v = vc.shape[2]
    k = idx.shape[-1]
    out = np.empty((B, T, H_q, d_v), np.uint16)
    lse = np.empty((B, T, H_q), np.float32)
    _load().oracle_sparse_attn_e4m3kv(_p(q), _p(kc), kc.shape[1] * d_qk, _p(ks), ks.shape[1],
                                      _p(vc), vc.shape[1] * d_v, _p(vs), vs.shape[1],
                                      _p(seq_len), _p(idx), B, T, H_q, d_qk, d_v, P, k,
                                      float(scale), _p(out), _p(lse))
    return out, lse


def i8_value(code: int, scale: float) -> float:
    return _load().oracle_i8_value(int(code), float(scale))


def i8_from_double(x: float, scale: float) -> int:
    """Nearest integer to x / scale in [-127, 127], ties to even."""
    return int(_load().oracle_i8_from_double(float(x), float(scale)))


def quantize_rows_i8(x):
    """bf16 rows [..., d] -> (int8 codes [..., d], fp32 scale per row = amax/127)."""
    x = _c(x, np.uint16)
    d = x.shape[-1]
    rows = int(np.prod(x.shape[:-1]))
    code = np.empty(x.shape, np.int8)
    scale = np.empty(x.shape[:-1], np.float32)
    _load().oracle_quantize_rows_i8(_p(x), rows, d, _p(code), _p(scale))
    return code, scale


def sparse_attn_i8kv(q, kc, ks, vc, vs, seq_len, idx, P, scale):
    """Attention over an INT8 K/V cache: element = code * the token row's
    scale.  kc [B][L][d_qk], vc [B][L][d_v] int8 codes; ks, vs [B][L] fp32."""
    q = _c(q, np.uint16)
    kc, vc = _c(kc, np.int8), _c(vc, np.int8)
    ks, vs = _c(ks, np.float32), _c(vs, np.float32)
    seq_len = _c(seq_len, np.int32)
    idx = _c(idx, np.int32)
    B, T, H_q, d_qk = q.shape
    d_v = vc.shape[2]
    k = idx.shape[-1]
    out = np.empty((B, T, H_q, d_v), np.uint16)
    lse = np.empty((B, T, H_q), np.float32)
    _load().oracle_sparse_attn_i8kv(_p(q), _p(kc), kc.shape[1] * d_qk, _p(ks), ks.shape[1],
                                    _p(vc), vc.shape[1] * d_v, _p(vs), vs.shape[1],
                                    _p(seq_len), _p(idx), B, T, H_q, d_qk, d_v, P, k,
                                    float(scale), _p(out), _p(lse))
    return out, lse


def index_scores_e4m3(cq, sq, w_head, ck, sk, seq_len, P, q_pos=None):
    """FP8 indexer score: sum_h w_h relu(sq_h sk_g sum_i v(cq) v(ck)); -inf if not visible.

    cq [B][T][H_i][d] and ck [B][G_max][d] are e4m3 codes with one fp32 scale
    per row (sq [B][T][H_i], sk [B][G_max])."""
    cq = _c(cq, np.uint8)
    ck = _c(ck, np.uint8)
    sq = _c(sq, np.float32)
    sk = _c(sk, np.float32)
    w_head = _c(w_head, np.float32)
    seq_len = _c(seq_len, np.int32)
    B, T, H_i, d = cq.shape
    G_max = ck.shape[1]
    qp = None if q_pos is None else _c(q_pos, np.int32)
    out = np.empty((B, T, G_max), np.float32)
    _load().oracle_index_scores_e4m3(_p(cq), _p(sq), _p(w_head), _p(ck), _p(sk), G_max * d,
                                     _p(seq_len), _p(qp), B, T, H_i, d, P, G_max, _p(out))
    return out


def topk(scores, n_valid, k):
    """Top-k visible groups per row (ties -> lower index), ascending, -1 padded."""
    scores = _c(scores, np.float32)
    n_valid = _c(n_valid, np.int32)
    G_max = scores.shape[-1]
    rows = int(np.prod(scores.shape[:-1]))
    assert n_valid.size == rows
    out = np.empty(scores.shape[:-1] + (k,), np.int32)
    _load().oracle_topk(_p(scores), _p(n_valid), rows, G_max, k, _p(out))
    return out


def sparse_attn(q, K, V, seq_len, idx, P, scale):
    """Attention of every query head over the tokens of the selected groups."""
    q = _c(q, np.uint16)
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    seq_len = _c(seq_len, np.int32)
    idx = _c(idx, np.int32)
    B, T, H_q, d_qk = q.shape
    d_v = V.shape[2]
    k = idx.shape[-1]
    out = np.empty((B, T, H_q, d_v), np.uint16)
    lse = np.empty((B, T, H_q), np.float32)
    _load().oracle_sparse_attn(_p(q), _p(K), K.shape[1] * d_qk, _p(V), V.shape[1] * d_v,
                               _p(seq_len), _p(idx), B, T, H_q, d_qk, d_v, P, k, float(scale),
                               _p(out), _p(lse))
    return out, lse


def retrieval_step(q_idx, w_head, k_pooled, q, K, V, seq_len, P, k, scale, q_pos=None):
    """score -> select -> attend over already pooled keys.

    Returns dict(scores, idx, out, lse).
    """
    q_idx = _c(q_idx, np.uint16)
    w_head = _c(w_head, np.float32)
    k_pooled = _c(k_pooled, np.uint16)
    q = _c(q, np.uint16)
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    seq_len = _c(seq_len, np.int32)
    qp = None if q_pos is None else _c(q_pos, np.int32)
    B, T, H_i, d_idx = q_idx.shape
    H_q, d_qk = q.shape[2], q.shape[3]
    d_v = V.shape[2]
    G_max = k_pooled.shape[1]
    scores = np.empty((B, T, G_max), np.float32)
    idx = np.empty((B, T, k), np.int32)
    out = np.empty((B, T, H_q, d_v), np.uint16)
    lse = np.empty((B, T, H_q), np.float32)
    _load().oracle_retrieval_step(_p(q_idx), _p(w_head), _p(k_pooled), G_max * d_idx, _p(q),
                                  _p(K), K.shape[1] * d_qk, _p(V), V.shape[1] * d_v,
                                  _p(seq_len), _p(qp), B, T, H_i, d_idx, P, G_max, k, H_q, d_qk,
                                  d_v, float(scale), _p(scores), _p(idx), _p(out), _p(lse))
    return dict(scores=scores, idx=idx, out=out, lse=lse)


def decode_case(case: dict, k_pooled=None):
    """Oracle of one generated workload (synth.generate output): pool, then step."""
    if k_pooled is None:
        k_pooled = pool_keys(case["k_idx"], case["pool_w"], case["seq_len"], case["P"])
    r = retrieval_step(case["q_idx"], case["w_head"], k_pooled, case["q"], case["K"], case["V"],
                       case["seq_len"], case["P"], case["k"], case["scale"], case["q_pos"])
    r["k_pooled"] = k_pooled
    return r
