"""KDA step on the GPU against the oracle (fp64 recurrence).

Tolerances, from the arithmetic (fp32 in the kernel, fp64 in the oracle):
  conv history   bit-exact (raw bf16 inputs are moved, not recomputed)
  state          |S_gpu - S_ref| <= 2e-6 * (1 + t) * max|S_ref| per head after
                 t tokens: each token rounds the decay product and the rank-one
                 update once (2^-24 relative each) on top of column sums over
                 128 channels whose errors enter through beta * k
  out (bf16)     |o_gpu - o_ref| <= 2^-8 |o_ref| + 2^-16 M_j, with
                 M_j = sum_i |q_i| |S'_ij| + |q.k| |beta (v_j - u_j)| the
                 magnitude of the terms the kernel sums in fp32 for o_j: one
                 bf16 rounding (2^-9 relative) plus fp32 sums over 128
                 channels (at most about 130 * 2^-24 * M_j; 2^-16 leaves a
                 factor of two)
"""
import numpy as np
import pytest
import torch

import long_context_sparse_weighted_b300 as lcsw
import oracle.kda as okda
import synth
import synth.kda as skda
from gpu_util import dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def _upload(c):
    return dict(qkv=dev_bf16(c["qkv"]), conv_w=dev_bf16(c["conv_w"]),
                conv_state=dev_bf16(c["conv_state"]), g=dev(c["g"]), beta=dev(c["beta"]),
                state=dev(c["state"]))


def _run(d, out=None):
    o = lcsw.kda_step(d["qkv"], d["conv_w"], d["conv_state"], d["g"], d["beta"], d["state"],
                      out=out)
    torch.cuda.synchronize()
    return o


def _bf16_f64(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


def _check(c, d, o, ref, T):
    o_ref, S_ref, cs_ref, M = ref
    got_o = _bf16_f64(host_bits(o))
    got_S = d["state"].cpu().numpy().astype(np.float64)
    got_cs = host_bits(d["conv_state"])
    assert np.array_equal(got_cs, cs_ref), "conv history differs"
    smax = np.abs(S_ref).max(axis=(-2, -1), keepdims=True)
    serr = np.abs(got_S - S_ref) / np.maximum(smax, 1e-30)
    assert serr.max() <= 2e-6 * (1 + T), f"state error {serr.max():.3g} x head max"
    bound = 2.0 ** -8 * np.abs(o_ref) + 2.0 ** -16 * M
    ratio = np.abs(got_o - o_ref) / np.maximum(bound, 1e-300)
    assert ratio.max() <= 1.0, f"{(ratio > 1).sum()} outputs off, worst at {ratio.max():.3g} x bound"
    return ratio.max()


def _oracle(c):
    """The oracle token by token, with the magnitude M of the terms summed for
    each output (the bound's second part)."""
    B, T, H, D = c["qkv"].shape[0], c["qkv"].shape[1], c["H"], c["D"]
    S = np.array(c["state"], dtype=np.float64)
    cs = c["conv_state"]
    o = np.zeros((B, T, H, D))
    M = np.zeros((B, T, H, D))
    for t in range(T):
        o_t, S_new, cs, parts = okda.kda_step(c["qkv"][:, t:t + 1], c["conv_w"], cs,
                                              c["g"][:, t:t + 1], c["beta"][:, t:t + 1], S, H, D,
                                              return_parts=True)
        q, k, v = parts[:, 0, 0], parts[:, 0, 1], parts[:, 0, 2]
        Sp = np.exp(np.asarray(c["g"][:, t], np.float64))[..., None] * S
        u = np.einsum("bhi,bhij->bhj", k, Sp)
        dw = np.asarray(c["beta"][:, t], np.float64)[..., None] * (v - u)
        qk = np.abs((q * k).sum(-1))[..., None]
        M[:, t] = np.einsum("bhi,bhij->bhj", np.abs(q), np.abs(Sp)) + qk * np.abs(dw)
        o[:, t] = o_t[:, 0]
        S = S_new
    return o, S, cs, M


@pytest.mark.parametrize("B,T,H", [(3, 1, 4), (2, 5, 3), (1, 2, 64)])
def test_kda_step_matches_oracle(B, T, H):
    c = skda.generate(skda.KdaSpec(B=B, T=T, H=H, D=128, seed=20 + B + T))
    ref = _oracle(c)
    d = _upload(c)
    o = _run(d)
    _check(c, d, o, ref, T)


def test_tokens_in_one_call_equal_single_token_calls():
    """The state stays fp32 between tokens in both cases, so the bits agree."""
    c = skda.generate(skda.KdaSpec(B=2, T=6, H=5, D=128, seed=30))
    d_all = _upload(c)
    o_all = _run(d_all)
    d = _upload(c)
    for t in range(c["T"]):
        sub = dict(d, qkv=d["qkv"][:, t:t + 1].contiguous(), g=d["g"][:, t:t + 1].contiguous(),
                   beta=d["beta"][:, t:t + 1].contiguous())
        o_t = _run(sub)
        assert torch.equal(o_t[:, 0].view(torch.int16), o_all[:, t].view(torch.int16))
    assert torch.equal(d["state"], d_all["state"])
    assert torch.equal(d["conv_state"].view(torch.int16), d_all["conv_state"].view(torch.int16))


def test_no_decay_no_write_keeps_the_state_exactly():
    c = skda.generate(skda.KdaSpec(B=2, T=3, H=4, D=128, seed=31))
    c["g"][:] = 0.0
    c["beta"][:] = 0.0
    d = _upload(c)
    before = d["state"].clone()
    o = _run(d)
    assert torch.equal(d["state"], before)
    ref = _oracle(c)
    _check(c, d, o, ref, c["T"])


def test_extreme_gates():
    """Full decay on some channels (alpha = exp(-80)), beta 0 and 1, and a
    head whose inputs are all zero (q = k = 0 after SiLU: the norm's epsilon
    keeps it finite)."""
    c = skda.generate(skda.KdaSpec(B=2, T=2, H=4, D=128, seed=32))
    c["g"][0, :, 0, :64] = -80.0
    c["beta"][0, :, 1] = 1.0
    c["beta"][1, :, 2] = 0.0
    HD = c["H"] * c["D"]
    for part in range(3):
        c["qkv"][1, :, part * HD + 3 * 128: part * HD + 4 * 128] = 0
        c["conv_state"][1, :, part * HD + 3 * 128: part * HD + 4 * 128] = 0
    ref = _oracle(c)
    d = _upload(c)
    o = _run(d)
    assert torch.isfinite(d["state"]).all()
    _check(c, d, o, ref, c["T"])


@pytest.mark.slow
def test_full_size_decode_step_sampled():
    """The benchmarked shape (64 sequences x 64 heads x 128 x 128 state, one
    token) in one call; the oracle checks two whole sequences."""
    spec = skda.named("kda_decode_b64")
    c = skda.generate(spec)
    d = _upload(c)
    o = _run(d)
    for b in (0, spec.B - 1):
        sub = {k: (v[b:b + 1] if isinstance(v, np.ndarray) and k != "conv_w" else v)
               for k, v in c.items()}
        o_ref, S_ref, cs_ref, M = _oracle(sub)
        got_o = _bf16_f64(host_bits(o[b:b + 1]))
        got_S = d["state"][b:b + 1].cpu().numpy().astype(np.float64)
        assert np.array_equal(host_bits(d["conv_state"][b:b + 1]), cs_ref)
        smax = np.abs(S_ref).max(axis=(-2, -1), keepdims=True)
        assert (np.abs(got_S - S_ref) / smax).max() <= 4e-6
        assert (np.abs(got_o - o_ref) <= 2.0 ** -8 * np.abs(o_ref) + 2.0 ** -16 * M).all()
