"""Seeded synthetic inputs for the pooled-indexer sparse-attention path.

This module only *draws inputs*: it holds none of the method's arithmetic
(no pooling, scoring, selection or attention).  Both the CUDA library's tests
and the CPU oracle are fed from here, so that the two sides see identical
bytes.

Random streams: numpy's Philox counter-based generator, keyed by
``(seed, tensor_id << 32 | chunk)``.  Every tensor is filled in fixed-size
chunks, each chunk from its own key, so the bytes do not depend on how many
threads generate them.

Workload recipes (the five named configurations) follow the release notes'
DSA layer description (page "G2C Brief — GLM-5.3-Flash", section "DSA keeps
selected global access in eleven layers": ``index_kpool: 4``,
``index_topk: 2048``) with synthetic value distributions:

* ``tiny``       B=1, L=4096, 4 indexer heads, integer-valued bf16 in [-3, 3],
                 head weights in {0.25, 0.5}, dyadic pool weights
                 (0.5, 0.25, 0.125, 0.125), top-k 64 groups, 16 query heads,
                 d=128, seed 0.
* ``decode_b8``  B=8, L=131072, 8 indexer heads N(0,1), softmax pool weights
                 from N(0,1) logits, top-k 512, 32 query heads,
                 d_qk=192 / d_v=128, scale 1/sqrt(192), seed 1.
* ``decode_1m``  B=1, L=1048576, 8 indexer heads N(0,1), 5% of raw keys get a
                 +3 sigma planted alignment to the query, top-k 512,
                 64 query heads, d=128, seed 2.
* ``ragged_b64`` B=64, L_b log-uniform in [8192, 262144] rounded to a
                 multiple of 4, top-k min(512, L_b/4), 32 query heads, d=128,
                 seed 3.
* ``prefill_4k`` B=1, 4096 new query tokens after 262144 cached tokens,
                 top-k 512 per query, 32 query heads, d=128, seed 4.
* ``mla_decode_1m`` decode_1m's indexer recipe with the MLA latent cache:
                 one 576-wide key row per token (latent 512 + rotary 64) whose
                 first 512 dims are the value, 64 query heads, seed 5.

Indexer head weights of the Gaussian workloads are U(0, 1) (the pages give
no distribution for them).  bf16 values are stored as their raw uint16 bit
patterns (round-to-nearest-even from float32).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

_CHUNK = 1 << 22  # elements per independently keyed chunk

# tensor ids (stable: changing one changes the bytes of that tensor only)
_TID = {
    "k_idx": 1, "pool_logits": 2, "q_idx": 3, "w_head": 4, "q": 5, "K": 6,
    "V": 7, "lengths": 8, "plant_pos": 9, "pool_w": 10,
}


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), round to nearest, ties to even.

    Inputs are finite; this is how the generator stores its draws.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern (uint16) -> float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, tid: int, chunk: int) -> np.random.Generator:
    key = np.array([seed & 0xFFFFFFFFFFFFFFFF, (tid << 32) | chunk], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def _fill(n: int, seed: int, tid: int, draw) -> np.ndarray:
    """Fill n values chunk by chunk; ``draw(rng, count)`` returns one chunk."""
    nchunks = (n + _CHUNK - 1) // _CHUNK
    parts = [None] * nchunks

    def one(i):
        cnt = min(_CHUNK, n - i * _CHUNK)
        parts[i] = draw(_rng(seed, tid, i), cnt)

    if nchunks <= 1:
        for i in range(nchunks):
            one(i)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(one, range(nchunks)))
    return np.concatenate(parts) if parts else np.zeros(0)


def normal_f32(n: int, seed: int, tid: int) -> np.ndarray:
    return _fill(n, seed, tid, lambda g, c: g.standard_normal(c, dtype=np.float32))


def normal_bf16(n: int, seed: int, tid: int) -> np.ndarray:
    return _fill(n, seed, tid,
                 lambda g, c: bf16_bits(g.standard_normal(c, dtype=np.float32)))


def int_bf16(n: int, lo: int, hi: int, seed: int, tid: int) -> np.ndarray:
    """Integers uniform in {lo, ..., hi} stored as bf16 (exact)."""
    return _fill(n, seed, tid, lambda g, c: bf16_bits(
        g.integers(lo, hi + 1, size=c).astype(np.float32)))


def uniform_f32(n: int, lo: float, hi: float, seed: int, tid: int) -> np.ndarray:
    return _fill(n, seed, tid, lambda g, c: g.uniform(lo, hi, size=c).astype(np.float32))


# ---------------------------------------------------------------------------
# workload description
# ---------------------------------------------------------------------------

@dataclass
class Spec:
    """Shape and value recipe of one synthetic workload."""
    name: str = "custom"
    B: int = 1
    lengths: Optional[list] = None   # total tokens per sequence (incl. new chunk)
    T: int = 1                       # query tokens per sequence
    prefill: bool = False            # queries are the last T tokens, causal at group level
    H_i: int = 8
    d_idx: int = 64
    P: int = 4
    k: int = 512                     # groups selected per query
    H_q: int = 32
    d_qk: int = 128
    d_v: int = 128
    scale: Optional[float] = None    # default 1/sqrt(d_qk)
    idx_values: str = "normal"       # "normal" | "int3"
    w_mode: str = "uniform01"        # "uniform01" | "quarter_half" | "onehot:<h>"
    pool_mode: str = "softmax"       # "softmax" | "dyadic" | "uniform" | "onehot:<j>"
    plant_frac: float = 0.0          # fraction of raw indexer keys planted toward q
    seed: int = 0
    L_cap: Optional[int] = None      # allocated tokens per sequence (>= max length)
    mla: bool = False                # one K row per token whose first d_v dims are V

    @property
    def L_max(self) -> int:
        lm = max(self.lengths)
        if self.L_cap is not None:
            lm = max(lm, self.L_cap)
        return lm

    @property
    def G_max(self) -> int:
        return self.L_max // self.P

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d_qk)


def ragged_lengths(B: int, lo: int, hi: int, seed: int, multiple: int = 4) -> list:
    """Log-uniform lengths in [lo, hi], rounded to a multiple of ``multiple``."""
    g = _rng(seed, _TID["lengths"], 0)
    u = g.uniform(math.log(lo), math.log(hi), size=B)
    out = []
    for x in u:
        L = int(round(math.exp(x) / multiple)) * multiple
        out.append(min(max(L, lo), hi))
    return out


def named(name: str) -> Spec:
    """The five named workloads."""
    if name == "tiny":
        return Spec(name=name, B=1, lengths=[4096], H_i=4, k=64, H_q=16, d_qk=128, d_v=128,
                    idx_values="int3", w_mode="quarter_half", pool_mode="dyadic", seed=0)
    if name == "decode_b8":
        return Spec(name=name, B=8, lengths=[131072] * 8, H_i=8, k=512, H_q=32, d_qk=192,
                    d_v=128, seed=1)
    if name == "decode_1m":
        return Spec(name=name, B=1, lengths=[1048576], H_i=8, k=512, H_q=64, d_qk=128,
                    d_v=128, plant_frac=0.05, seed=2)
    if name == "ragged_b64":
        return Spec(name=name, B=64, lengths=ragged_lengths(64, 8192, 262144, 3), H_i=8,
                    k=512, H_q=32, d_qk=128, d_v=128, seed=3)
    if name == "mla_decode_1m":
        # decode_1m's indexer and selection with the MLA latent cache: one
        # 576-wide row per token (latent 512 + rotary 64), the latent as value
        return Spec(name=name, B=1, lengths=[1048576], H_i=8, k=512, H_q=64, d_qk=576,
                    d_v=512, plant_frac=0.05, mla=True, seed=5)
    if name == "prefill_4k":
        return Spec(name=name, B=1, lengths=[262144 + 4096], T=4096, prefill=True, H_i=8,
                    k=512, H_q=32, d_qk=128, d_v=128, seed=4)
    raise KeyError(name)


NAMES = ("tiny", "decode_b8", "decode_1m", "ragged_b64", "prefill_4k")


def shrink(spec: Spec, factor: int, min_len: int = 1024) -> Spec:
    """Same recipe with every context length divided by ``factor`` (multiple of P)."""
    lens = [max(min_len, (L // factor) // spec.P * spec.P) for L in spec.lengths]
    T = min(spec.T, max(1, min(lens) // 2)) if spec.prefill else spec.T
    return replace(spec, lengths=lens, T=T, name=spec.name + f"/{factor}")


# ---------------------------------------------------------------------------
# generation
# ---------------------------------------------------------------------------

def _pool_weights(spec: Spec, G_max: int) -> np.ndarray:
    P = spec.P
    B = spec.B
    mode = spec.pool_mode
    if mode == "dyadic":
        row = [2.0 ** -(j + 1) for j in range(P - 1)] + [2.0 ** -(P - 1)]
        return np.broadcast_to(np.array(row, np.float32), (B, G_max, P)).copy()
    if mode == "uniform":
        return np.full((B, G_max, P), 1.0 / P, np.float32)
    if mode.startswith("onehot:"):
        j = int(mode.split(":")[1])
        w = np.zeros((B, G_max, P), np.float32)
        w[:, :, j] = 1.0
        return w
    if mode == "softmax":
        z = normal_f32(B * G_max * P, spec.seed, _TID["pool_logits"]).astype(np.float64)
        z = z.reshape(B, G_max, P)
        z = z - z.max(axis=2, keepdims=True)
        e = np.exp(z)
        return (e / e.sum(axis=2, keepdims=True)).astype(np.float32)
    if mode == "random":  # arbitrary positive weights, not normalised
        return uniform_f32(B * G_max * P, 0.0, 1.0, spec.seed,
                           _TID["pool_w"]).reshape(B, G_max, P)
    raise ValueError(mode)


def _head_weights(spec: Spec) -> np.ndarray:
    n = spec.B * spec.T * spec.H_i
    if spec.w_mode == "uniform01":
        w = uniform_f32(n, 0.0, 1.0, spec.seed, _TID["w_head"])
    elif spec.w_mode == "quarter_half":
        g = _fill(n, spec.seed, _TID["w_head"], lambda r, c: r.integers(0, 2, size=c))
        w = np.where(g == 0, 0.25, 0.5).astype(np.float32)
    elif spec.w_mode == "signed":
        w = normal_f32(n, spec.seed, _TID["w_head"])
    elif spec.w_mode.startswith("onehot:"):
        h = int(spec.w_mode.split(":")[1])
        w = np.zeros(n, np.float32).reshape(spec.B, spec.T, spec.H_i)
        w[:, :, h] = 1.0
        return w
    else:
        raise ValueError(spec.w_mode)
    return w.reshape(spec.B, spec.T, spec.H_i)


def generate(spec: Spec, with_kv: bool = True) -> dict:
    """Draw every input of one workload.

    Returns a dict of numpy arrays (bf16 as uint16 bit patterns):
      seq_len [B] int32, q_pos [B][T] int32 or None,
      k_idx [B][L_max][d_idx], pool_w [B][G_max][P] f32,
      q_idx [B][T][H_i][d_idx], w_head [B][T][H_i] f32,
      q [B][T][H_q][d_qk], K [B][L_max][d_qk], V [B][L_max][d_v]
    plus the scalar parameters.  Tokens at or past seq_len[b] are zero.
    """
    B, T, P = spec.B, spec.T, spec.P
    L_max, G_max = spec.L_max, spec.G_max
    lens = np.array(spec.lengths, dtype=np.int32)
    assert len(lens) == B and (lens >= 0).all() and (lens <= L_max).all()
    s = spec.seed

    def per_token(tid, width, kind):
        out = np.zeros((B, L_max, width), np.uint16)
        # one stream per (tensor, sequence): draw only the valid tokens
        for b in range(B):
            n = int(lens[b]) * width
            if n == 0:
                continue
            sub = (tid << 8) | b
            if kind == "int3":
                v = int_bf16(n, -3, 3, s, sub)
            else:
                v = normal_bf16(n, s, sub)
            out[b, :lens[b]] = v.reshape(int(lens[b]), width)
        return out

    k_idx = per_token(_TID["k_idx"], spec.d_idx, spec.idx_values)
    n_qi = B * T * spec.H_i * spec.d_idx
    if spec.idx_values == "int3":
        q_idx = int_bf16(n_qi, -3, 3, s, _TID["q_idx"])
    else:
        q_idx = normal_bf16(n_qi, s, _TID["q_idx"])
    q_idx = q_idx.reshape(B, T, spec.H_i, spec.d_idx)

    if spec.plant_frac > 0:
        # Planted alignment: a fraction of raw token keys k_t gets
        # k_t <- bf16(k_t + 3*sqrt(H_i)*u), u = unit(sum_h q_h/|q_h|) of the
        # sequence's first query, which lifts each head's dot product by about
        # three standard deviations of q_h.k for k ~ N(0, I).
        qf = bf16_to_f32(q_idx).astype(np.float64)
        for b in range(B):
            Lb = int(lens[b])
            npl = int(spec.plant_frac * Lb)
            if npl == 0:
                continue
            qh = qf[b, 0]
            u = (qh / np.linalg.norm(qh, axis=1, keepdims=True)).sum(axis=0)
            u /= np.linalg.norm(u)
            shift = 3.0 * math.sqrt(spec.H_i) * u
            pos = _rng(s, _TID["plant_pos"], b).permutation(Lb)[:npl]
            pos.sort()
            kf = bf16_to_f32(k_idx[b, pos]).astype(np.float64) + shift[None, :]
            k_idx[b, pos] = bf16_bits(kf.astype(np.float32))

    pool_w = _pool_weights(spec, G_max)
    w_head = _head_weights(spec)
    q = normal_bf16(B * T * spec.H_q * spec.d_qk, s, _TID["q"]).reshape(B, T, spec.H_q, spec.d_qk)

    if spec.prefill:
        q_pos = np.stack([np.arange(int(lens[b]) - T, int(lens[b]), dtype=np.int32)
                          for b in range(B)])
        assert (q_pos >= 0).all()
    else:
        q_pos = None

    out = dict(spec=spec, seq_len=lens, q_pos=q_pos, k_idx=k_idx, pool_w=pool_w,
               q_idx=q_idx, w_head=w_head, q=q, B=B, T=T, P=P, L_max=L_max, G_max=G_max,
               H_i=spec.H_i, d_idx=spec.d_idx, k=spec.k, H_q=spec.H_q, d_qk=spec.d_qk,
               d_v=spec.d_v, scale=spec.softmax_scale)
    if with_kv:
        out["K"] = per_token(_TID["K"], spec.d_qk, "normal")
        if spec.mla:
            # the MLA latent geometry: the value is the latent part of the key row
            out["V"] = np.ascontiguousarray(out["K"][:, :, :spec.d_v])
        else:
            out["V"] = per_token(_TID["V"], spec.d_v, "normal")
    return out
