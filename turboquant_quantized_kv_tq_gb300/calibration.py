"""Host-side calibration of the SQU-KV codec (numpy; offline, not part of the decode or append).

For one side (K or V) of one KV head, from representative vectors X (n x d) of that side:
normalize each to a unit vector u; take the eigen-decomposition of mean(u u^T); return the
eigenvectors by descending eigenvalue as the basis E (columns), and the coordinate scales
s_j = sqrt(d lambda_j).  [ABL] "Configuração Experimental" (SpectralQuant's per-head basis
calibrated on representative tokens), "Recomendações Práticas" 2 (separate calibration sets for
K and V).  The spectral-gap effective dimension is returned for information: the built codec
models the top 32 directions at 4 bits and keeps 1 bit for the rest.
"""

import numpy as np

_FLOOR = 1e-12


def spectral_basis(X):
    """(E float32 [d][d], s float32 [d], d_eff) for QuantizedKVCache.set_spectral_basis."""
    X = np.asarray(X, dtype=np.float64)
    n = np.linalg.norm(X, axis=1)
    U = X[n > 0] / n[n > 0, None]
    w, V = np.linalg.eigh(U.T @ U / U.shape[0])
    order = np.argsort(-w, kind="stable")
    lam = np.clip(w[order], 0.0, None)
    d = X.shape[1]
    floor = np.maximum(lam, _FLOOR * lam[0])
    d_eff = int(np.argmax(floor[:-1] / floor[1:])) + 1
    s = np.maximum(np.sqrt(d * lam), np.sqrt(d * _FLOOR * lam[0]))
    return V[:, order].astype(np.float32), s.astype(np.float32), d_eff


def spectral_tables(calib):
    """Stacked tables of every KV head: calib [H_kv][n][d] -> (E [H_kv][d][d], s [H_kv][d],
    d_eff per head)."""
    out = [spectral_basis(calib[h]) for h in range(len(calib))]
    return np.stack([o[0] for o in out]), np.stack([o[1] for o in out]), [o[2] for o in out]
