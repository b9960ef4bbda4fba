"""The synthetic workloads follow the stated input recipe (CPU).

Shapes of the named workloads, integer-valued and dyadic tiny inputs, softmax
pool weights, the ragged length law, the planted 5 % of decode_1m, zero tokens
past each length, and bit-identical regeneration from a seed.
"""
import numpy as np

import synth


def test_named_shapes():
    for name, (B, L, H_i, k, H_q, d_qk, d_v) in {
            "tiny": (1, 4096, 4, 64, 16, 128, 128),
            "decode_b8": (8, 131072, 8, 512, 32, 192, 128),
            "decode_1m": (1, 1048576, 8, 512, 64, 128, 128)}.items():
        s = synth.named(name)
        assert (s.B, max(s.lengths), s.H_i, s.k, s.H_q, s.d_qk, s.d_v, s.P, s.d_idx) == \
            (B, L, H_i, k, H_q, d_qk, d_v, 4, 64), name
    assert abs(synth.named("decode_b8").softmax_scale - 192 ** -0.5) < 1e-12


def test_ragged_lengths_law():
    L = np.array(synth.named("ragged_b64").lengths)
    assert len(L) == 64 and (L % 4 == 0).all()
    assert L.min() >= 8192 and L.max() <= 262144
    # log-uniform on [8192, 262144]: the logs' mean is the log of the geometric mean
    assert abs(np.log(L).mean() - 0.5 * (np.log(8192) + np.log(262144))) < 0.35


def test_tiny_values():
    c = synth.generate(synth.named("tiny"))
    k = synth.bf16_to_f32(c["k_idx"][0, :4096])
    q = synth.bf16_to_f32(c["q_idx"])
    for x in (k, q):
        assert set(np.unique(x)) <= set(range(-3, 4)) and len(np.unique(x)) == 7
    assert set(np.unique(c["w_head"])) <= {0.25, 0.5}
    assert np.array_equal(c["pool_w"][0, 0], np.array([0.5, 0.25, 0.125, 0.125], np.float32))


def test_softmax_pool_weights_and_zero_tail():
    s = synth.shrink(synth.named("ragged_b64"), 64)
    c = synth.generate(s)
    w = c["pool_w"].astype(np.float64)
    assert (w > 0).all() and np.allclose(w.sum(axis=2), 1.0, atol=1e-6)
    for b in range(s.B):
        Lb = int(c["seq_len"][b])
        assert not c["k_idx"][b, Lb:].any() and not c["K"][b, Lb:].any()
        assert c["k_idx"][b, :Lb].any()


def test_planted_fraction_lifts_scores():
    s = synth.shrink(synth.named("decode_1m"), 64)
    base = synth.generate(synth.Spec(**{**s.__dict__, "plant_frac": 0.0}), with_kv=False)
    c = synth.generate(s, with_kv=False)
    changed = (c["k_idx"][0] != base["k_idx"][0]).any(axis=1)
    L = int(c["seq_len"][0])
    assert changed.sum() <= int(0.05 * L) and changed.sum() >= int(0.05 * L) - 2
    # the planted keys score higher against the query, head by head
    q = synth.bf16_to_f32(c["q_idx"][0, 0]).astype(np.float64)     # [H_i][64]
    k = synth.bf16_to_f32(c["k_idx"][0]).astype(np.float64)        # [L][64]
    dots = k @ q.T
    assert (dots[changed].mean(axis=0) > dots[~changed].mean(axis=0) + 2.0 *
            np.linalg.norm(q, axis=1)).all()


def test_regeneration_is_bit_identical():
    s = synth.shrink(synth.named("decode_b8"), 64)
    a, b = synth.generate(s), synth.generate(s)
    for key in ("k_idx", "pool_w", "q_idx", "w_head", "q", "K", "V"):
        assert np.array_equal(a[key], b[key]), key
    other = synth.generate(synth.Spec(**{**s.__dict__, "seed": s.seed + 1}))
    assert not np.array_equal(a["K"], other["K"])


def test_kda_recipe():
    import synth.kda as skda
    s = skda.named("kda_decode_b64")
    assert (s.B, s.T, s.H, s.D) == (64, 1, 64, 128)
    c = skda.generate(skda.KdaSpec(B=2, T=3, H=4, D=128, seed=11))
    C = 3 * 4 * 128
    assert c["qkv"].shape == (2, 3, C) and c["conv_w"].shape == (C, 4)
    assert c["conv_state"].shape == (2, 3, C) and c["state"].shape == (2, 4, 128, 128)
    g, beta = c["g"], c["beta"]
    assert (g <= 0).all() and (g >= -0.25).all()          # alpha = e^g in [0.78, 1]
    assert (beta >= 0).all() and (beta <= 1).all()
    w = synth.bf16_to_f32(c["conv_w"])
    assert (np.abs(w) <= 0.5).all()
    assert abs(c["state"].std() - 0.05) < 0.005
