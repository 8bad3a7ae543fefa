"""Seeded constant tables: rotation signs D and QJL sketch matrix S (float64 then fp32).

The pages fix no random-number generator ([ABL] "Configuração Experimental" even
validates an oracle and a GPU build that use different generators).  Bit-exact
codes need both sides to hold the very same D and S, so each side implements
one published counter-based generator from its definition:

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): state advances by the golden-ratio increment
  0x9E3779B97F4A7C15 and each output is the 64-bit finalizer ``mix64`` of
  the state.  Stream ``s`` of seed ``seed`` starts from state
  ``seed XOR mix64(s)``; draw ``i`` (0-based) is ``mix64(state + (i+1)*gamma)``.
* Streams: D_K = 1, D_V = 2, S_K = 3, S_V = 4.
* D_i = +1 when the top bit of draw i of its stream is 0, else -1.
* S (m x d, row-major, entry n = i*d + j) is the cosine branch of Box-Muller
  on draws 2n and 2n+1: u1 = ((h1 >> 11) + 1) * 2^-53 in (0, 1],
  u2 = (h2 >> 11) * 2^-53 in [0, 1),
  S = sqrt(-2 ln u1) * cos(6.283185307179586 * u2) in float64 with the C
  library's scalar log / cos / sqrt, then rounded to fp32 (nearest even).
"""

import math

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15

STREAM_D_K = 1
STREAM_D_V = 2
STREAM_S_K = 3
STREAM_S_V = 4


def mix64(z):
    """SplitMix64 output finalizer on a Python int (mod 2**64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def draws(seed, stream, count):
    """The first ``count`` draws of stream ``stream`` as a list of Python ints."""
    state = (seed ^ mix64(stream)) & MASK64
    out = []
    for i in range(count):
        out.append(mix64((state + (i + 1) * GAMMA) & MASK64))
    return out


def rotation_signs(seed, stream, d):
    """D as a float64 vector of +-1 (top bit 0 -> +1)."""
    return np.array([1.0 if (h >> 63) == 0 else -1.0 for h in draws(seed, stream, d)])


def sketch_matrix(seed, stream, m, d):
    """S (m x d) with i.i.d. N(0, 1) entries, fp32, from Box-Muller on consecutive draws."""
    h = draws(seed, stream, 2 * m * d)
    out = np.empty(m * d, dtype=np.float32)
    two_pi = 6.283185307179586
    for n in range(m * d):
        u1 = ((h[2 * n] >> 11) + 1) * 2.0 ** -53
        u2 = (h[2 * n + 1] >> 11) * 2.0 ** -53
        out[n] = np.float32(math.sqrt(-2.0 * math.log(u1)) * math.cos(two_pi * u2))
    return out.reshape(m, d)
