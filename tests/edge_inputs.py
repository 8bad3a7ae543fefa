"""Hand-built inputs for the method's edge cases (test infrastructure; no codec arithmetic).

* ``tie_vectors``: fp32 vectors of exact unit norm whose first nonzero coordinate equals a given
  fp32 value exactly, so that under Plain-KV (no rotation) y = x / ||x|| lands exactly on a
  decision threshold.  The remaining mass 1 - t^2 is written as a sum of squares of fp32 values
  by a greedy integer square root in exact integer arithmetic.
* ``extreme_vectors``: bf16-representable vectors whose sums of squares overflow or underflow
  fp32, or that mix huge and tiny coordinates.
"""

import math
from fractions import Fraction

import numpy as np

from workloads import bf16_bits


def _dyadic(t):
    """fp32 value t as (m, f) with t = m / 2^f exactly (m an integer)."""
    fr = Fraction(float(np.float32(t)))
    f = fr.denominator.bit_length() - 1
    assert fr.denominator == 1 << f
    return fr.numerator, f


def unit_remainder_squares(t):
    """fp32 values a_1.. (as float32) with t^2 + sum a_i^2 = 1 exactly, |t| < 1."""
    m, f = _dyadic(t)
    f = max(f, 12)  # at least 2^-12 resolution for the remainder
    N = (1 << (2 * f)) - m * m * (1 << (2 * f - 2 * _dyadic(t)[1]))
    assert N >= 0
    out = []
    while N > 0:
        a = math.isqrt(N)
        a = (a >> max(0, a.bit_length() - 24)) << max(0, a.bit_length() - 24)  # 24 significant bits
        N -= a * a
        out.append(a)
    vals = [np.float32(Fraction(a, 1 << f)) for a in out]
    assert all(Fraction(float(v)) == Fraction(a, 1 << f) for v, a in zip(vals, out)), "not exact in fp32"
    return vals


def tie_vectors(targets, d, positions):
    """One vector per (target, position): x[pos] = target, the greedy remainder in the next
    coordinates (cyclically), zeros elsewhere; every vector has sum x^2 = 1 exactly."""
    rows = []
    for t in targets:
        for pos in positions:
            x = np.zeros(d, dtype=np.float32)
            x[pos] = np.float32(t)
            rem = unit_remainder_squares(t)
            assert len(rem) < d - 1
            for i, a in enumerate(rem):
                x[(pos + 1 + i) % d] = a
            rows.append(x)
    return np.stack(rows)


def exact_square_sum(x):
    return sum(Fraction(float(v)) ** 2 for v in np.asarray(x, dtype=np.float32).ravel())


def extreme_vectors(rng, n, d):
    """bf16 bit patterns [n][d] cycling through five kinds of vector:
    0: one coordinate near the bf16 maximum, the rest of order 1e-30;
    1: every coordinate of order 1e19 (the fp32 sum of squares overflows);
    2: every coordinate of order 1e-25 (every square underflows fp32);
    3: coordinates of order 1e-20 (squares in the fp32 subnormal range);
    4: a vector of order 1 with a few coordinates near 1e-38."""
    X = np.empty((n, d), dtype=np.float64)
    for i in range(n):
        kind = i % 5
        g = rng.standard_normal(d)
        if kind == 0:
            X[i] = 1e-30 * g
            X[i, rng.integers(d)] = (2.5e38 if rng.random() < 0.5 else -2.5e38) * (0.5 + 0.5 * rng.random())
        elif kind == 1:
            X[i] = 1e19 * g
        elif kind == 2:
            X[i] = 1e-25 * g
        elif kind == 3:
            X[i] = 1e-20 * g
        else:
            X[i] = g
            X[i, rng.integers(d, size=4)] = 1e-38 * rng.standard_normal(4)
    return bf16_bits(X.astype(np.float32))
