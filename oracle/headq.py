"""HeadQ calibration basis and corrected logits (float64).

[HEADQ] "Visão Geral do Algoritmo":
  1. calibration: a rank-r basis U_h per head learned by PCA of calibration
     queries;
  3. read: s_hat_j = q^T k_base_j / sqrt(d) + q^T U_h z_hat_j / sqrt(d).

Readings: the basis is per KV head (the side code is stored once per key, so
the G query heads of a group share it), and it is the top-r eigenvectors of
the centred sample covariance of that group's calibration queries.

``calibration_basis`` is pinned by tests/test_oracle_headq_basis.py through
what is unique about it (eigenvector signs and degenerate subspaces are not):
the projector onto a planted subspace, orthonormality, maximal captured
variance (Ky Fan) against other frames, invariance to a common offset and to
scale, and the leading direction by brute force at d = 2.  It is calibration
input handed identically to both sides as an fp32 table and never compared.
"""

import numpy as np


def calibration_basis(queries, rank):
    """Top-``rank`` principal directions (d x rank) of calibration queries (N x d)."""
    Q = np.asarray(queries, dtype=np.float64)
    Qc = Q - Q.mean(axis=0, keepdims=True)
    cov = Qc.T @ Qc / max(Q.shape[0] - 1, 1)
    w, v = np.linalg.eigh(cov)
    order = np.argsort(w)[::-1][:rank]
    return v[:, order]


def corrected_logits(q, kbase, U, side, side_scale):
    """s_hat_j = q^T k_base_j / sqrt(d) + q^T U z_hat_j / sqrt(d), z_hat = scale * zeta."""
    d = q.shape[-1]
    zhat = np.asarray(side_scale, dtype=np.float64)[:, None] * np.asarray(side, dtype=np.float64)
    return (kbase @ q + zhat @ (np.asarray(U, dtype=np.float64).T @ q)) / np.sqrt(d)
