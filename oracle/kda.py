"""CPU oracle of the KDA decode step (the linear-attention half of the hybrid).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use this module; the CUDA library never
imports or calls it and shares no code with it.

What the pages fix (page "G2C Brief -- GLM-5.3-Flash", section "KDA carries
fixed state through most layers"): Kimi Delta Attention is a gated delta-rule
descendant of linear attention that keeps a fixed matrix state per head
instead of a growing K/V cache; a short convolution of kernel size 4 and
learned gates surround the recurrence; the config has 64 heads of width 128,
so the state is 64 x 128 x 128 values per layer.  The pages print no formula.
The readings taken here (the plainest that the text supports, stated once so
a reader can check them):

1. Recurrence, per head, with S the D_k x D_v state (key channels as rows):
       S' = Diag(alpha_t) S_{t-1}                       (channel-wise decay gate)
       S_t = (I - beta_t k_t k_t^T) S' + beta_t k_t v_t^T   (delta-rule write)
       o_t = S_t^T q_t
   alpha_t = exp(g_t) per key channel, beta_t in [0, 1] per head.
2. Short convolution: depthwise and causal over the q, k and v channels,
   kernel 4, no bias, each output through SiLU (x * sigmoid(x)).  Tap 3
   multiplies the current token, tap 0 the token three steps back.
3. q and k are L2-normalised per head after the convolution,
   x / sqrt(sum x^2 + 1e-6); q is then scaled by D_k^-1/2.
4. The gates arrive as inputs (g = log alpha <= 0 and beta); their
   projections, like the q/k/v projections and the output gate and norm,
   are dense layers of the model and lie outside the step.

Arithmetic is fp64 throughout; bf16 inputs are widened exactly.
"""
from __future__ import annotations

import numpy as np

L2_EPS = 1e-6
CONV_K = 4


def bf16_to_f64(b) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exact."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x), written so that neither branch overflows."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = x[pos] / (1.0 + np.exp(-x[pos]))
    e = np.exp(x[~pos])
    out[~pos] = x[~pos] * e / (1.0 + e)
    return out


def short_conv(window: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Depthwise causal convolution at one token (reading 2).

    window: [4][C], the inputs of tokens t-3, t-2, t-1, t per channel;
    w: [C][4], tap j multiplying window[j].  Returns the pre-activation [C].
    """
    return np.einsum("jc,cj->c", window, w)


def l2_normalize(x: np.ndarray) -> np.ndarray:
    """x / sqrt(sum x^2 + eps) along the last axis (reading 3)."""
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2_EPS)


def delta_rule_update(S: np.ndarray, q: np.ndarray, k: np.ndarray, v: np.ndarray,
                      alpha: np.ndarray, beta: float):
    """One gated delta-rule step of one head (reading 1).

    S [D_k][D_v], q and k [D_k] (q already scaled), v [D_v], alpha [D_k].
    Returns (S_t, o_t).
    """
    Sp = alpha[:, None] * S
    eye = np.eye(S.shape[0])
    S_new = (eye - beta * np.outer(k, k)) @ Sp + beta * np.outer(k, v)
    return S_new, S_new.T @ q


def kda_step(qkv, conv_w, conv_state, g, beta, state, H: int, D: int, return_parts=False):
    """T tokens of the KDA step for B sequences.

    qkv        [B][T][3*H*D] bf16 bits: pre-convolution q | k | v, head-major.
    conv_w     [3*H*D][4] bf16 bits.
    conv_state [B][3][3*H*D] bf16 bits: inputs of the three previous tokens,
               oldest first.
    g          [B][T][H][D] fp32, log decay per key channel; beta [B][T][H].
    state      [B][H][D][D] float, rows = key channels.

    Returns (o [B][T][H][D] fp64, new state [B][H][D][D] fp64,
    new conv_state [B][3][3*H*D] uint16); with return_parts also the
    activated, normalised q (scaled), k and v of every token.
    """
    qkv = np.asarray(qkv, dtype=np.uint16)
    B, T, C = qkv.shape
    assert C == 3 * H * D
    w = bf16_to_f64(conv_w).reshape(C, CONV_K)
    S = np.array(state, dtype=np.float64).reshape(B, H, D, D)
    cs = np.array(conv_state, dtype=np.uint16).reshape(B, CONV_K - 1, C)
    g = np.asarray(g, dtype=np.float64).reshape(B, T, H, D)
    beta = np.asarray(beta, dtype=np.float64).reshape(B, T, H)
    o = np.zeros((B, T, H, D))
    parts = np.zeros((B, T, 3, H, D))
    scale = 1.0 / np.sqrt(D)
    for b in range(B):
        hist = [cs[b, j] for j in range(CONV_K - 1)]  # bf16 bits, oldest first
        for t in range(T):
            window = np.stack([bf16_to_f64(x) for x in hist + [qkv[b, t]]])
            act = silu(short_conv(window, w)).reshape(3, H, D)
            q = l2_normalize(act[0]) * scale
            k = l2_normalize(act[1])
            v = act[2]
            parts[b, t] = np.stack([q, k, v])
            for h in range(H):
                S[b, h], o[b, t, h] = delta_rule_update(S[b, h], q[h], k[h], v[h],
                                                        np.exp(g[b, t, h]), beta[b, t, h])
            hist = hist[1:] + [qkv[b, t]]
        cs[b] = np.stack(hist)
    if return_parts:
        return o, S, cs, parts
    return o, S, cs
