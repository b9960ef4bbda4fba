"""Pins of the KDA oracle against things other than itself.

The hand-worked fixture (tests/golden/kda_worked.txt), properties the delta
rule fixes by its algebra (a write along k leaves every direction orthogonal
to k untouched and moves the read-out along k to (1 - beta) old + beta v),
library routines for the special cases (np.convolve for the causal
convolution, scipy's expit for the sigmoid) and brute-force equivalences
(T tokens in one call = T single-token calls).  Planted mistakes in a copy of
the oracle must each fail one of the pins.
"""
import types

import numpy as np
import pytest
from scipy.special import expit

import oracle.kda as kda
import synth
import synth.kda as skda
from conftest import read_fixture


def _f(vals):
    return np.array([float(x) for x in vals])


# ---------------------------------------------------------------------------
# the planted-mistake harness: a copy of the module with one edit
# ---------------------------------------------------------------------------

MUTANTS = {
    # decay applied after the delta-rule write instead of before
    "decay_after_write": ("    Sp = alpha[:, None] * S\n    eye = np.eye(S.shape[0])\n"
                          "    S_new = (eye - beta * np.outer(k, k)) @ Sp + beta * np.outer(k, v)\n",
                          "    Sp = S\n    eye = np.eye(S.shape[0])\n"
                          "    S_new = alpha[:, None] * ((eye - beta * np.outer(k, k)) @ Sp"
                          " + beta * np.outer(k, v))\n"),
    # decay over value columns instead of key channels
    "decay_on_columns": ("Sp = alpha[:, None] * S", "Sp = S * alpha[None, :]"),
    # read-out through S instead of S^T
    "readout_untransposed": ("return S_new, S_new.T @ q", "return S_new, S_new @ q"),
    # erase term dropped (plain gated linear attention)
    "no_erase": ("(eye - beta * np.outer(k, k)) @ Sp", "Sp"),
    # state read before the write
    "readout_before_write": ("return S_new, S_new.T @ q", "return S_new, Sp.T @ q"),
    # conv taps reversed
    "taps_reversed": ('np.einsum("jc,cj->c", window, w)', 'np.einsum("jc,cj->c", window[::-1], w)'),
    # SiLU dropped
    "no_silu": ("act = silu(short_conv(window, w))", "act = short_conv(window, w)"),
    # q not scaled
    "q_unscaled": ("q = l2_normalize(act[0]) * scale", "q = l2_normalize(act[0])"),
    # k not normalised
    "k_unnormalised": ("k = l2_normalize(act[1])", "k = act[1]"),
    # conv history not advanced
    "history_frozen": ("hist = hist[1:] + [qkv[b, t]]", "hist = hist"),
    # gate taken as alpha itself instead of log alpha
    "gate_not_exp": ("np.exp(g[b, t, h])", "g[b, t, h]"),
}


def _mutant(name):
    old, new = MUTANTS[name]
    src = open(kda.__file__).read()
    assert src.count(old) == 1, name
    mod = types.ModuleType(f"kda_{name}")
    exec(compile(src.replace(old, new), f"kda_{name}", "exec"), mod.__dict__)
    return mod


def _pins(mod):
    """Every pin below, run against `mod`; returns the names that fail."""
    failed = []
    for fn in PINS:
        try:
            fn(mod)
        except (AssertionError, ValueError):   # a wrong shape counts as a failed pin
            failed.append(fn.__name__)
    return failed


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_worked_delta_step(m):
    fx = read_fixture("kda_worked.txt")
    S = np.stack([_f(fx["S0"]), _f(fx["S1"])])
    S_new, o = m.delta_rule_update(S, _f(fx["q"]), _f(fx["k"]), _f(fx["v"]), _f(fx["alpha"]),
                                   float(fx["beta"][0]))
    np.testing.assert_allclose(S_new, np.stack([_f(fx["expect_S0"]), _f(fx["expect_S1"])]),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, _f(fx["expect_o"]), rtol=0, atol=1e-12)


def pin_worked_recall(m):
    fx = read_fixture("kda_worked.txt")
    S = np.zeros((2, 2))
    one = np.ones(2)
    S, _ = m.delta_rule_update(S, one, _f(fx["r_k1"]), _f(fx["r_v1"]), one, 1.0)
    S, o = m.delta_rule_update(S, _f(fx["r_q"]), _f(fx["r_k2"]), _f(fx["r_v2"]), one, 1.0)
    np.testing.assert_allclose(S, np.stack([_f(fx["r_expect_S0"]), _f(fx["r_expect_S1"])]),
                               atol=1e-12)
    np.testing.assert_allclose(o, _f(fx["r_expect_o"]), atol=1e-12)


def pin_worked_conv(m):
    fx = read_fixture("kda_worked.txt")
    y = m.short_conv(_f(fx["c_x"])[:, None], _f(fx["c_w"])[None, :])
    assert abs(y[0] - float(fx["c_expect"][0])) < 1e-12


def pin_write_algebra(m):
    """Random S, alpha, beta, unit k, non-square state: along k the read-out
    becomes (1 - beta) S'^T k + beta v; orthogonal to k nothing changes."""
    rng = np.random.default_rng(5)
    Dk, Dv = 7, 5
    S = rng.standard_normal((Dk, Dv))
    alpha = rng.uniform(0.2, 1.0, Dk)
    k = rng.standard_normal(Dk)
    k /= np.linalg.norm(k)
    v = rng.standard_normal(Dv)
    beta = 0.3
    S_new, _ = m.delta_rule_update(S, np.zeros(Dk), k, v, alpha, beta)
    Sp = np.diag(alpha) @ S
    np.testing.assert_allclose(S_new.T @ k, (1 - beta) * (Sp.T @ k) + beta * v, atol=1e-12)
    z = rng.standard_normal(Dk)
    z -= (z @ k) * k
    np.testing.assert_allclose(S_new.T @ z, Sp.T @ z, atol=1e-12)


def pin_readout_is_state_transpose(m):
    """o = S_t^T q: the read-out is linear in q and, for q = e_i, row i of S_t."""
    rng = np.random.default_rng(6)
    Dk, Dv = 6, 3
    S = rng.standard_normal((Dk, Dv))
    k = np.eye(Dk)[2]
    for i in range(Dk):
        S_new, o = m.delta_rule_update(S, np.eye(Dk)[i], k, np.ones(Dv), np.ones(Dk), 0.5)
        np.testing.assert_allclose(o, S_new[i], atol=1e-12)


def pin_full_decay_wipes(m):
    """alpha = 0 everywhere: S_t = beta k v^T, o = beta (k.q) v."""
    rng = np.random.default_rng(7)
    D = 8
    k = rng.standard_normal(D)
    k /= np.linalg.norm(k)
    q, v = rng.standard_normal(D), rng.standard_normal(D)
    S_new, o = m.delta_rule_update(rng.standard_normal((D, D)), q, k, v, np.zeros(D), 0.7)
    np.testing.assert_allclose(S_new, 0.7 * np.outer(k, v), atol=1e-12)
    np.testing.assert_allclose(o, 0.7 * (k @ q) * v, atol=1e-12)


def pin_silu_is_x_times_sigmoid(m):
    x = np.array([-80.0, -3.5, -1e-3, 0.0, 1e-3, 2.0, 40.0])
    np.testing.assert_allclose(m.silu(x), x * expit(x), rtol=1e-15, atol=0)


def pin_conv_matches_np_convolve(m):
    """A channel driven from a zero history: the pre-activation sequence is the
    causal convolution with the taps in reverse (np.convolve's kernel order)."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal(12)
    w = rng.standard_normal(4)
    hist = [0.0, 0.0, 0.0]
    got = []
    for t in range(len(x)):
        window = np.array(hist + [x[t]])[:, None]
        got.append(m.short_conv(window, w[None, :])[0])
        hist = hist[1:] + [x[t]]
    np.testing.assert_allclose(got, np.convolve(x, w[::-1])[:len(x)], atol=1e-12)


def _small_case(seed=12, T=4):
    return skda.generate(skda.KdaSpec(B=2, T=T, H=3, D=16, seed=seed))


def pin_step_parts(m):
    """The activated parts of a whole step: q and k unit length (times the
    scale for q, up to the epsilon), v = SiLU of the convolution, each checked
    against its definition written independently here with expit."""
    c = _small_case()
    H, D = c["H"], c["D"]
    _, _, _, parts = m.kda_step(c["qkv"], c["conv_w"], c["conv_state"], c["g"], c["beta"],
                                c["state"], H, D, return_parts=True)
    w = synth.bf16_to_f32(c["conv_w"]).astype(np.float64)
    x = synth.bf16_to_f32(c["qkv"]).astype(np.float64)
    h0 = synth.bf16_to_f32(c["conv_state"]).astype(np.float64)
    for b in range(c["B"]):
        seq = np.concatenate([h0[b], x[b]])          # [3 + T][C]
        for t in range(c["T"]):
            y = sum(w[:, j] * seq[t + j] for j in range(4))
            a = (y * expit(y)).reshape(3, H, D)
            nq = np.sqrt((a[0] ** 2).sum(-1, keepdims=True) + 1e-6)
            nk = np.sqrt((a[1] ** 2).sum(-1, keepdims=True) + 1e-6)
            np.testing.assert_allclose(parts[b, t, 0], a[0] / nq / np.sqrt(D), rtol=1e-12,
                                       atol=1e-15)
            np.testing.assert_allclose(parts[b, t, 1], a[1] / nk, rtol=1e-12, atol=1e-15)
            np.testing.assert_allclose(parts[b, t, 2], a[2], rtol=1e-12, atol=1e-15)


def pin_step_state_along_k(m):
    """Whole step, beta = 1 and no decay: afterwards S^T k = v for the token's
    own (normalised) key and v, and o = S^T q."""
    c = _small_case(T=1)
    c["beta"][:] = 1.0
    c["g"][:] = 0.0
    H, D = c["H"], c["D"]
    o, S, _, parts = m.kda_step(c["qkv"], c["conv_w"], c["conv_state"], c["g"], c["beta"],
                                c["state"], H, D, return_parts=True)
    for b in range(c["B"]):
        for h in range(H):
            q, k, v = parts[b, 0, 0, h], parts[b, 0, 1, h], parts[b, 0, 2, h]
            kn = k / np.linalg.norm(k)      # |k| = 1 up to the epsilon
            np.testing.assert_allclose(S[b, h].T @ kn, v, atol=1e-6 * np.abs(v).max())
            np.testing.assert_allclose(o[b, 0, h], S[b, h].T @ q, atol=1e-12)


def pin_tokens_split_across_calls(m):
    """T tokens in one call = T calls of one token each (conv history and
    state handed over between calls)."""
    c = _small_case(T=5)
    H, D = c["H"], c["D"]
    o_all, S_all, cs_all = m.kda_step(c["qkv"], c["conv_w"], c["conv_state"], c["g"],
                                      c["beta"], c["state"], H, D)
    S, cs = c["state"], c["conv_state"]
    for t in range(c["T"]):
        o_t, S, cs = m.kda_step(c["qkv"][:, t:t + 1], c["conv_w"], cs, c["g"][:, t:t + 1],
                                c["beta"][:, t:t + 1], S, H, D)
        np.testing.assert_allclose(o_t[:, 0], o_all[:, t], atol=1e-12)
    np.testing.assert_allclose(S, S_all, atol=1e-12)
    assert np.array_equal(cs, cs_all)


def pin_conv_history_is_last_inputs(m):
    """After a call the conv history holds the raw inputs of the last three
    tokens, oldest first (bit for bit: they are stored, not recomputed)."""
    c = _small_case(T=5)
    _, _, cs = m.kda_step(c["qkv"], c["conv_w"], c["conv_state"], c["g"], c["beta"],
                          c["state"], c["H"], c["D"])
    assert np.array_equal(cs, c["qkv"][:, -3:])


def pin_gate_is_log_decay(m):
    """g = log 0.5 on every channel with beta = 0: one step halves the state;
    g = 0 keeps it."""
    c = _small_case(T=1)
    c["beta"][:] = 0.0
    c["g"][:] = np.float32(np.log(0.5))
    _, S, _ = m.kda_step(c["qkv"], c["conv_w"], c["conv_state"], c["g"], c["beta"],
                         c["state"], c["H"], c["D"])
    np.testing.assert_allclose(S, 0.5 * c["state"].astype(np.float64), rtol=1e-6)
    c["g"][:] = 0.0
    _, S, _ = m.kda_step(c["qkv"], c["conv_w"], c["conv_state"], c["g"], c["beta"],
                         c["state"], c["H"], c["D"])
    np.testing.assert_allclose(S, c["state"].astype(np.float64), rtol=0, atol=0)


PINS = [pin_worked_delta_step, pin_worked_recall, pin_worked_conv, pin_write_algebra,
        pin_readout_is_state_transpose, pin_full_decay_wipes, pin_silu_is_x_times_sigmoid,
        pin_conv_matches_np_convolve, pin_step_parts, pin_step_state_along_k,
        pin_tokens_split_across_calls, pin_conv_history_is_last_inputs, pin_gate_is_log_decay]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(kda)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    failed = _pins(_mutant(name))
    assert failed, f"mutant {name} passes every pin"
