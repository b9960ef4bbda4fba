"""Seeded synthetic inputs for the KDA (gated delta-rule) decode step.

Draws inputs only: none of the recurrence, the convolution or the gates'
arithmetic lives here.  The CUDA tests, the bench and the CPU oracle all take
their bytes from these functions.

Geometry follows the release's linear-attention config (page "G2C Brief --
GLM-5.3-Flash", section "KDA carries fixed state through most layers"): 64
heads of width 128, so a 64 x 128 x 128 matrix state per sequence and layer,
and a short convolution of kernel size 4.  The pages give no value
distributions; the recipe here is:

* ``qkv``       pre-convolution q, k and v projections, N(0, 1) in bf16;
                per token one row of 3*H*D values ordered q | k | v, each
                part head-major.
* ``conv_w``    depthwise conv taps, U(-0.5, 0.5) in bf16, [3*H*D][4],
                tap 3 multiplying the current token.
* ``conv_state`` the previous three inputs of every channel, N(0, 1) in bf16,
                [3][3*H*D] (oldest first).
* ``g``         log of the per-key-channel decay, -U(0, 0.25) in fp32 (so
                alpha = exp(g) lies in [0.78, 1]).
* ``beta``      per-head write strength, U(0, 1) in fp32.
* ``state``     the recurrent matrix state, N(0, 0.05^2) in fp32, [H][D][D]
                (key channel rows, value columns).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import normal_bf16, normal_f32, uniform_f32, _fill, bf16_bits

_TID = {"qkv": 40, "conv_w": 41, "conv_state": 42, "g": 43, "beta": 44, "state": 45}


@dataclass
class KdaSpec:
    B: int = 64          # sequences
    T: int = 1           # tokens per call (1 = one decode step)
    H: int = 64          # heads
    D: int = 128         # head width (key and value)
    seed: int = 10


def named(name: str) -> KdaSpec:
    if name == "kda_decode_b64":
        return KdaSpec(B=64, T=1, H=64, D=128, seed=10)
    if name == "kda_tiny":
        return KdaSpec(B=2, T=3, H=4, D=128, seed=11)
    raise KeyError(name)


def _uniform_bf16(n, lo, hi, seed, tid):
    return _fill(n, seed, tid, lambda g, c: bf16_bits(g.uniform(lo, hi, size=c).astype(np.float32)))


def generate(spec: KdaSpec) -> dict:
    """Inputs of one KDA step over spec.T tokens for spec.B sequences."""
    B, T, H, D, s = spec.B, spec.T, spec.H, spec.D, spec.seed
    C = 3 * H * D
    out = dict(B=B, T=T, H=H, D=D)
    out["qkv"] = normal_bf16(B * T * C, s, _TID["qkv"]).reshape(B, T, C)
    out["conv_w"] = _uniform_bf16(C * 4, -0.5, 0.5, s, _TID["conv_w"]).reshape(C, 4)
    out["conv_state"] = normal_bf16(B * 3 * C, s, _TID["conv_state"]).reshape(B, 3, C)
    out["g"] = -uniform_f32(B * T * H * D, 0.0, 0.25, s, _TID["g"]).reshape(B, T, H, D)
    out["beta"] = uniform_f32(B * T * H, 0.0, 1.0, s, _TID["beta"]).reshape(B, T, H)
    st = normal_f32(B * H * D * D, s, _TID["state"]) * np.float32(0.05)
    out["state"] = st.astype(np.float32).reshape(B, H, D, D)
    return out
