"""SpectralQuant with uniform bit allocation (SQU-KV) at 2 bits per coordinate, float64.
Test infrastructure only.

[ABL] "Configuração Experimental" describes SpectralQuant as a data-adaptive codec.  It
calibrates a per-head eigenvector basis from representative tokens and spends the bits on the
high-variance dimensions.  "Armazenamento vs. Qualidade" gives the unmodeled tail dimensions a
fixed floor.  "Recomendações Práticas" 2-3 keep the uniform-allocation variant (water-filling
brings nothing), with K and V calibrated on separate sets.  "Contribuições Principais" 3 sizes
the modeled dimension by a spectral-gap criterion.

Readings (the summary gives no formulas or sizes):

* Calibration works on the unit vectors u = x / ||x|| of a side's calibration set, because the
  codec quantizes u after the norm split.  M = mean(u u^T) is the uncentred second moment, so
  eigenvalue lambda_i is the mean square of coordinate i in the eigenbasis.  The basis E holds
  M's eigenvectors as columns, by descending eigenvalue.  d_eff is the k with the largest
  eigenvalue ratio lambda_k / lambda_(k+1) (eigenvalues floored at 1e-12 lambda_1); calibration
  reports it.
* Uniform allocation at 2 bits per coordinate (the budget of TQ-KV n=2): the TOP = 32
  highest-variance directions are modeled at 4 bits each, and the 96 others keep a 1-bit floor.
  The storage (256 bits per vector) is the same as TQ-KV n=2's.  A calibration with d_eff > 32
  is truncated to the top 32.
* Scale: coordinate i's value z_i = (E^T u)_i / s_i with s_i = sqrt(d lambda_i) has the mean
  square 1/d of a sphere coordinate.  The 4-bit and 1-bit Beta Lloyd-Max codebooks of the
  TurboQuant path (dimension d) then quantize it unchanged.  The decision compares fp32(z) with
  the fp32 thresholds.
* Storage order: coordinate c of the stored vector is an eigen-rank chosen so that the modeled
  coordinates form whole pieces of the decoder's operands.  Keys: ranks 0..31 go to
  coordinates 32 (i % 4) + i // 4, the first 8 of each 32-coordinate chunk.  Values: rank i
  goes to 16 (i % 8) + i // 8, the first 4 of each 16-coordinate group.  The tail ranks fill the
  other coordinates in increasing order.  E and s are stored in that order (E[:, c], s[c]).
* A code record (32 bytes at d = 128) is a 4-bit stream of the modeled coordinates' magnitudes,
  in increasing coordinate order (sign-magnitude form of the 4-bit code; the 1-bit codebook has
  a magnitude of one level), followed by a 1-bit stream of every coordinate's sign (1 =
  positive).  On the value side both streams are stored by 16-coordinate groups like every
  value stream (oracle/layout.py): a group holds the 4 magnitudes (2 bytes) or 16 signs
  (2 bytes) of one group of coordinates.
"""

import numpy as np

from . import codec, layout

TOP = 32
TOP_BITS = 4
FLOOR_BITS = 1
EIG_FLOOR = 1e-12


def unit_rows(X):
    X = np.asarray(X, dtype=np.float64)
    n = np.sqrt(np.sum(X * X, axis=1))
    keep = n > 0
    return X[keep] / n[keep, None]


def effective_dim(lam):
    """argmax_k lambda_k / lambda_(k+1), k in [1, d - 1] (1-based count of modeled dims)."""
    lam = np.asarray(lam, dtype=np.float64)
    f = np.maximum(lam, EIG_FLOOR * lam[0])
    return int(np.argmax(f[:-1] / f[1:])) + 1


def calibrate(X):
    """(E, lam, d_eff): eigenvectors of mean(u u^T) as columns (descending eigenvalues)."""
    U = unit_rows(X)
    M = U.T @ U / U.shape[0]
    w, V = np.linalg.eigh(M)
    order = np.argsort(-w, kind="stable")
    lam = np.maximum(w[order], 0.0)
    return V[:, order], lam, effective_dim(lam)


def rank_of_coord(side, d=128):
    """Eigen-rank stored at each coordinate (see the storage-order reading)."""
    rank = np.full(d, -1, dtype=np.int64)
    for i in range(TOP):
        c = 32 * (i % 4) + i // 4 if side == "k" else 16 * (i % 8) + i // 8
        rank[c] = i
    tail = [c for c in range(d) if rank[c] < 0]
    rank[tail] = np.arange(TOP, d)
    return rank


def top_mask(side, d=128):
    return rank_of_coord(side, d) < TOP


def rank_tables(E, lam):
    """(E32, s32) in eigen-rank order, rounded to fp32 once: s_j = sqrt(d lambda_j), floored."""
    d = E.shape[0]
    lam = np.asarray(lam, dtype=np.float64)
    s = np.maximum(np.sqrt(d * lam), np.sqrt(d * EIG_FLOOR * lam[0]))
    return np.asarray(E, dtype=np.float32), np.asarray(s, dtype=np.float32)


def storage_tables(E, lam, side):
    """(E32, s32): the basis and scales in storage order (a permutation of rank_tables; the
    tables both sides use)."""
    E32, s32 = rank_tables(E, lam)
    r = rank_of_coord(side, E32.shape[0])
    return E32[:, r], s32[r]


def encode(X, side, E32, s32, C4, T4, C1, T1):
    """Codes of vectors X (N x d): z = (E^T u) / s in float64 from the fp32 tables; modeled
    coordinates take the 4-bit code of fp32(z), the others the 1-bit code.  Returns norm (fp32),
    codes (ascending index in each coordinate's own codebook), z and the decision margin."""
    X = np.asarray(X, dtype=np.float64)
    nu = np.sqrt(np.sum(X * X, axis=1))
    safe = np.where(nu > 0, nu, 1.0)
    u = np.where(nu[:, None] > 0, X / safe[:, None], 0.0)
    z = (u @ np.asarray(E32, dtype=np.float64)) / np.asarray(s32, dtype=np.float64)[None, :]
    top = top_mask(side, X.shape[1])
    c4, c1 = codec.quantize_codes(z, T4), codec.quantize_codes(z, T1)
    m4, m1 = codec.boundary_distance(z, T4), codec.boundary_distance(z, T1)
    return {"norm": nu.astype(np.float32), "codes": np.where(top, c4, c1), "z": z,
            "code_margin": np.where(top, m4, m1)}


def reconstruct(codes, norm32, side, E32, s32, C4, C1):
    """x_hat = nu E (s * C[c]), each coordinate through its own codebook."""
    top = top_mask(side, np.asarray(codes).shape[1])
    zhat = np.where(top, np.asarray(C4, dtype=np.float64)[np.minimum(codes, len(C4) - 1)],
                    np.asarray(C1, dtype=np.float64)[np.minimum(codes, len(C1) - 1)])
    zs = zhat * np.asarray(s32, dtype=np.float64)[None, :]
    return norm32.astype(np.float64)[:, None] * (zs @ np.asarray(E32, dtype=np.float64).T)


def pack(codes, side):
    """Code records (N x d/4 bytes): magnitudes of the modeled coordinates, then every sign."""
    codes = np.asarray(codes, dtype=np.int64)
    top = top_mask(side, codes.shape[1])
    sgn = np.where(top, codes >= (1 << (TOP_BITS - 1)), codes >= 1).astype(np.int64)
    _, mag = layout.to_sign_magnitude(codes[:, top], TOP_BITS)
    return np.concatenate([layout.pack_stream(mag, 4), layout.pack_stream(sgn, 1)], axis=1)


def unpack(data, side, d=128):
    top = top_mask(side, d)
    data = np.asarray(data, dtype=np.uint8)
    mag = layout.unpack_stream(data[:, : TOP // 2], 4, TOP)
    sgn = layout.unpack_stream(data[:, TOP // 2:], 1, d)
    codes = sgn.copy()  # floor coordinates: the 1-bit code is the sign
    codes[:, top] = layout.from_sign_magnitude(sgn[:, top], mag & 7, TOP_BITS)
    return codes
