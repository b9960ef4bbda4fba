"""Hard inputs for the pooled-key sum: weights and keys built so that the exact
sum sum_j alpha_j * k_j lies exactly on a bf16 rounding midpoint, a hair to
either side of one, after a cancellation of large terms, or spans very
different magnitudes.  Only input construction lives here (fp32 weights, bf16
bit patterns, and the exact rational sum for checking), shared by the oracle
pins and the GPU parity test.
"""
from fractions import Fraction

import numpy as np


def f32(x):
    return np.float32(x)


def bf16_bits(x):
    """bf16 bit pattern of a value that is exactly representable in bf16."""
    b = int(np.array([x], np.float32).view(np.uint32)[0])
    assert b & 0xFFFF == 0, f"{x} is not a bf16 value"
    return b >> 16


def bf16_val(bits):
    return float(np.array([int(bits) << 16], np.uint32).view(np.float32)[0])


def round_bf16(x: Fraction) -> int:
    """Nearest bf16 of an exact rational (ties to even), from the format: 8
    significant bits, subnormal quantum 2^-133, overflow to infinity."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    qe = max(e - 7, -133)
    r = a / Fraction(2) ** qe
    n = r.numerator // r.denominator
    rem = r - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = Fraction(n) * Fraction(2) ** qe
    if v >= Fraction(2) ** 128:
        return sign | 0x7F80
    return sign | bf16_bits(float(v))


def exact_sum(alpha, kbits):
    return sum(Fraction(float(a)) * Fraction(bf16_val(k)) for a, k in zip(alpha, kbits))


def _rand_bf16(rng, lo=-20, hi=20):
    m = 1.0 + rng.integers(0, 128) / 128.0
    return float(np.ldexp(m, int(rng.integers(lo, hi)))) * (1 if rng.random() < 0.5 else -1)


def cases(n=400, seed=31, P=4):
    """n groups of (alpha[P] fp32, keys[P] bf16 bits)."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        kind = i % 4
        alpha = [f32(0.0)] * P
        keys = [0] * P
        if kind == 0:
            # v + ulp(v)/2 + delta: a bf16 midpoint, exactly or nudged by a tiny term
            v = abs(_rand_bf16(rng))
            ex = int(np.floor(np.log2(v)))
            half = 2.0 ** (ex - 8)
            alpha[0], keys[0] = f32(1.0), bf16_bits(v)
            alpha[1], keys[1] = f32(half), bf16_bits(1.0)
            if i % 8 != 0:
                tiny = 2.0 ** (ex - 8 - int(rng.integers(1, 60)))
                sgn = 1.0 if rng.random() < 0.5 else -1.0
                alpha[2], keys[2] = f32(tiny), bf16_bits(sgn)
        elif kind == 1:
            # two large terms cancel exactly; the rest decides (and may tie)
            a = f32(rng.uniform(0.1, 1.0))
            x = _rand_bf16(rng, 30, 60)
            alpha[0], keys[0] = a, bf16_bits(x)
            alpha[1], keys[1] = a, bf16_bits(-x)
            alpha[2], keys[2] = f32(rng.uniform(0.0, 1.0)), bf16_bits(_rand_bf16(rng, -10, 10))
            alpha[3], keys[3] = f32(np.ldexp(rng.uniform(0.5, 1.0), -40)), bf16_bits(
                _rand_bf16(rng, -10, 10))
        elif kind == 2:
            # wildly different magnitudes
            for j in range(P):
                alpha[j] = f32(np.ldexp(rng.uniform(0.5, 1.0), int(rng.integers(-120, 20))))
                keys[j] = bf16_bits(_rand_bf16(rng, -120, 100))
        else:
            # a softmax-like row with one tiny key beside large ones
            w = rng.dirichlet(np.ones(P)).astype(np.float32)
            for j in range(P):
                alpha[j] = f32(w[j])
                keys[j] = bf16_bits(_rand_bf16(rng, -3, 3))
            keys[P - 1] = bf16_bits(_rand_bf16(rng, -100, -60))
        out.append((np.array(alpha, np.float32), np.array(keys, np.uint16)))
    return out


def as_arrays(cs, d=64):
    """Pack cases into k_idx [1][P*G][d] and pool_w [1][G][P] (G = len(cs)); every
    dimension of group g holds case g."""
    P = len(cs[0][0])
    G = len(cs)
    k_idx = np.zeros((1, P * G, d), np.uint16)
    pool_w = np.zeros((1, G, P), np.float32)
    for g, (a, k) in enumerate(cs):
        pool_w[0, g] = a
        k_idx[0, P * g:P * g + P, :] = k[:, None]
    return k_idx, pool_w
