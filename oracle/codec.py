"""Per-vector encoder and reconstruction of the quantized KV cache (float64).

Schemes ([TQ-KV] "Esquemas de Cuantización"; [ABL] "Contribuições Principais" 1),
all at n bits per coordinate ([TQ-KV] "Esquemas de Cuantización": equal budget):

* Plain-KV: n-bit Lloyd-Max scalar code on K and V, no rotation, no sketch.
* TQ-KV:    rotation + n-bit code on K and V.
* KQV:      rotation; K n-bit code; V (n-1)-bit code + 1-bit QJL residual sketch.
* QKQV (also named TQ-QKV): rotation; K and V both (n-1)-bit code + 1-bit QJL.

Readings (the pages are summaries and leave these open):

* "n bits por vector" in [TQ-KV] means n bits per coordinate: the scheme list
  splits n into n-1 scalar bits plus a 1-bit sketch.
* The norm is split off first and stored as fp32; the unit vector is rotated
  and quantized (a unit vector's rotated coordinate follows the Beta marginal,
  [TQ-KV] "Marco Teórico").  Plain-KV uses the same norm split and codebook.
* QJL ([TQ-KV] "Contribuciones Clave" 1): the residual r = y - C[c] of the
  rotated unit vector is summarized by sign(S r) (S: m x d, N(0,1) entries)
  and ||r|| (stored fp16).  The unbiased estimate of <a, r> is
  sqrt(pi/2) / m * ||r|| * <S a, sign(S r)>, so the reconstruction adds
  r_hat = sqrt(pi/2) / m * ||r|| * S^T (2 sigma - 1).
* Ties: a coordinate exactly on a threshold takes the lower cell; a sketch
  coordinate (S r)_i = 0 gives sign bit 1.
* A zero vector has norm 0 and unit vector 0; its codes follow the tie rule
  (the middle threshold is 0, so every coordinate takes the cell just below
  it), its residual is -C[c] like any other vector's, and it reconstructs to
  0 because its norm is 0.
* A code decision compares the fp32 rounding of y against fp32 thresholds,
  the precision the decoder's tables hold.
* HeadQ ([HEADQ] "Visão Geral do Algoritmo" 2): base key k_base = B_b(k) from
  the K codec, e = k - k_base in the original key domain, z = U^T e with the
  calibrated basis U (d x r), side quantizer Q_q symmetric uniform with
  levels -7..7 (4 bits) and a per-key fp16 scale max|z| / 7; codes
  zeta = clamp(rint(z / s), -7, 7) with round-half-even, taken in fp32.
"""

from dataclasses import dataclass

import numpy as np

QJL_SCALE_NUM = np.sqrt(np.pi / 2.0)  # sqrt(pi/2); divided by m at use


@dataclass(frozen=True)
class SideCodec:
    bits: int
    rotate: bool
    qjl: bool
    spectral: bool = False  # SQU-KV (oracle/spectral.py): calibrated basis, 32 x 4 + 96 x 1 bits


def scheme_codecs(scheme, n):
    """(K codec, V codec) of a scheme at n bits per coordinate."""
    s = scheme.lower().replace("_", "-")
    if s in ("plain", "plain-kv", "kv"):
        return SideCodec(n, False, False), SideCodec(n, False, False)
    if s in ("tq", "tq-kv"):
        return SideCodec(n, True, False), SideCodec(n, True, False)
    if s == "kqv":
        if n < 2:
            raise ValueError("KQV needs n >= 2")
        return SideCodec(n, True, False), SideCodec(n - 1, True, True)
    if s in ("qkqv", "tq-qkv"):
        if n < 2:
            raise ValueError("QKQV needs n >= 2")
        return SideCodec(n - 1, True, True), SideCodec(n - 1, True, True)
    if s in ("squ", "squ-kv"):
        if n != 2:
            raise ValueError("SQU-KV is built at n = 2 (its record is TQ-KV n=2's size)")
        return SideCodec(2, False, False, True), SideCodec(2, False, False, True)
    raise ValueError("unknown scheme " + scheme)


def quantize_codes(y, thresholds32):
    """c_i = number of fp32 thresholds strictly below fp32(y_i) (ascending centroid index)."""
    y32 = np.asarray(y, dtype=np.float64).astype(np.float32)
    t = np.asarray(thresholds32, dtype=np.float32)
    return np.sum(y32[..., None] > t, axis=-1).astype(np.int64)


def boundary_distance(y, thresholds32):
    """min_k |y_i - t_k| in float64 against the fp32 thresholds (exempt zone measure)."""
    t = np.asarray(thresholds32, dtype=np.float32).astype(np.float64)
    return np.min(np.abs(np.asarray(y, dtype=np.float64)[..., None] - t), axis=-1)


def encode(x, codec, centroids32, thresholds32, R, S=None):
    """Encode vectors x (N x d, float64) with one side's codec.

    Returns a dict with norm (fp32), codes (ascending index), and for QJL sides
    rho (fp16) and signs (bool, m per vector), plus the float64 intermediates
    (y, Sr) that parity tests use to locate decision boundaries.
    """
    x = np.asarray(x, dtype=np.float64)
    nu = np.sqrt(np.sum(x * x, axis=1))
    nu32 = nu.astype(np.float32)
    safe = np.where(nu > 0, nu, 1.0)
    u = np.where(nu[:, None] > 0, x / safe[:, None], 0.0)
    y = u @ np.asarray(R, dtype=np.float64).T
    c = quantize_codes(y, thresholds32)
    out = {"norm": nu32, "codes": c, "y": y, "code_margin": boundary_distance(y, thresholds32)}
    if codec.qjl:
        r = y - np.asarray(centroids32, dtype=np.float64)[c]
        rho16 = np.sqrt(np.sum(r * r, axis=1)).astype(np.float16)
        Sr = r @ np.asarray(S, dtype=np.float64).T
        out.update({"rho": rho16, "signs": Sr >= 0.0, "Sr": Sr, "residual": r})
    return out


def headq_encode(x, codes, norm32, centroids32, R, U, side_bits=4):
    """HeadQ side code ([HEADQ] "Visão Geral do Algoritmo" 2, "Escrita no Cache").

    k_base = nu R^T C[c]; e = k - k_base; z = U^T e; s = fp16(max|z| / qmax);
    zeta = clamp(rint(z / s), -qmax, qmax), qmax = 2**(side_bits-1) - 1.
    """
    qmax = (1 << (side_bits - 1)) - 1
    x = np.asarray(x, dtype=np.float64)
    kbase = norm32.astype(np.float64)[:, None] * (np.asarray(centroids32, dtype=np.float64)[codes] @ R)
    e = x - kbase
    z = e @ np.asarray(U, dtype=np.float64)
    a = np.max(np.abs(z), axis=1) / qmax
    s16 = a.astype(np.float16)
    s32 = s16.astype(np.float32)
    zs = np.where(s32[:, None] > 0, z.astype(np.float32) / np.where(s32 > 0, s32, 1)[:, None], np.float32(0))
    zeta = np.clip(np.rint(zs), -qmax, qmax).astype(np.int64)
    # distance of z to the nearest rounding boundary s*(k + 1/2), in the key's units
    frac = np.abs(z / np.where(s32 > 0, s32, 1).astype(np.float64)[:, None])
    margin = np.abs(frac - (np.floor(frac) + 0.5)) * s32.astype(np.float64)[:, None]
    return {"side": zeta, "side_scale": s16, "z": z, "side_margin": margin,
            "scale_margin": fp16_midpoint_distance(a)}


def fp16_midpoint_distance(a):
    """Relative distance of each float64 value ``a`` to the nearest point where rounding to fp16
    changes (the midpoint between the two fp16 values around it); the exempt-zone measure of
    the HeadQ side scale, whose fp16 rounding is a decision like a code's."""
    a = np.asarray(a, dtype=np.float64)
    h = a.astype(np.float16)
    hf = h.astype(np.float64)
    other = np.where(hf <= a, np.nextafter(h, np.float16(np.inf)), np.nextafter(h, np.float16(-np.inf)))
    mid = (hf + other.astype(np.float64)) / 2.0
    return np.abs(a - mid) / np.where(a > 0, a, 1.0)


def reconstruct(codec, codes, norm32, centroids32, R, rho16=None, signs=None, S=None,
                side=None, side_scale=None, U=None):
    """x_hat = nu R^T (C[c] + r_hat) (+ U z_hat for HeadQ keys), from stored values."""
    yhat = np.asarray(centroids32, dtype=np.float64)[np.asarray(codes)]
    if codec.qjl:
        m = S.shape[0]
        pm = np.where(np.asarray(signs), 1.0, -1.0)
        yhat = yhat + (QJL_SCALE_NUM / m) * rho16.astype(np.float64)[:, None] * (pm @ np.asarray(S, dtype=np.float64))
    xhat = norm32.astype(np.float64)[:, None] * (yhat @ np.asarray(R, dtype=np.float64))
    if side is not None:
        zhat = side_scale.astype(np.float64)[:, None] * np.asarray(side, dtype=np.float64)
        xhat = xhat + zhat @ np.asarray(U, dtype=np.float64).T
    return xhat


def qjl_inner_product(a, S, rho, signs):
    """QJL estimate of <a, r>: sqrt(pi/2)/m * ||r|| * <S a, 2 sigma - 1> ([TQ-KV] "Contribuciones Clave" 1)."""
    S = np.asarray(S, dtype=np.float64)
    m = S.shape[0]
    pm = np.where(np.asarray(signs), 1.0, -1.0)
    return (QJL_SCALE_NUM / m) * rho * np.dot(S @ a, pm)
