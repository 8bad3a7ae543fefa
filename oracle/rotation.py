"""Seeded randomized Walsh-Hadamard rotation, as explicit matrices (float64).

[TQ-KV] "Esquemas de Cuantización" items 2-3 and [ABL] "Configuração
Experimental" (TurboQuant item) rotate K and V with a randomized Walsh-Hadamard
transform before scalar quantization.  The pages give no formula; the standard
form is used: y = H D x / sqrt(d), H the Sylvester Hadamard matrix in natural
order, H_ij = (-1)^popcount(i & j), D a seeded diagonal of +-1.  Plain-KV uses
no rotation ([TQ-KV] "Esquemas de Cuantización" item 1).
"""

import numpy as np


def sylvester_hadamard(d):
    """H_ij = (-1)^popcount(i & j) for a power of two d, built entry by entry."""
    if d <= 0 or d & (d - 1):
        raise ValueError("d must be a power of two")
    i = np.arange(d)
    parity = np.zeros((d, d), dtype=np.int64)
    both = i[:, None] & i[None, :]
    while np.any(both):
        parity ^= both & 1
        both = both >> 1
    return np.where(parity == 1, -1.0, 1.0)


def rotation_matrix(signs):
    """R = H diag(D) / sqrt(d), orthogonal."""
    d = len(signs)
    return sylvester_hadamard(d) * np.asarray(signs, dtype=np.float64)[None, :] / np.sqrt(d)
