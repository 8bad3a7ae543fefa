"""Seeded synthetic inputs of the five benchmark configurations.

This module only draws random inputs; it holds none of the codec's arithmetic, and both the
CUDA library's callers and the CPU oracle's callers take their inputs from here.  Draws use
numpy's PCG64 (``default_rng(seed)``) in the order K, V, q (then calibration queries),
slab by slab ([batch][KV head]) so that memory stays bounded at full size.  bf16 tensors are
returned as their uint16 bit patterns (round to nearest even from float32).

Configurations (the pages measure on no public dataset; these synthetic regimes stand in for
the pages' Gaussian, heavy-tailed, low-rank and outlier-channel distributions):

* ``cfg1``  1 head, d=128, T=1024, fp32 N(0,1) K, V, q; seed 0; TQ-KV n=4.
* ``cfg2``  B=8, H_q=32, H_kv=8, d=128, T=32768; K, V Student-t(3)/sqrt(3) in bf16; q N(0,1).
* ``cfg3``  B=4, H_q=H_kv=8, d=1024, T=8192; K = z U^T + eps (U a seeded orthonormal rank-16
            basis, z ~ N(0, I), eps ~ N(0, 0.01 I)); V ~ N(0,1); q = w U^T + eps'; bf16 K, V.
* ``cfg4``  B=1, H_q=64, H_kv=8, d=128, T=131072; Gaussian K, V with a per-(tensor, KV head,
            channel) std drawn log-uniform in [0.1, 10]; bf16; q N(0,1); 4096-token prefill chunk.
* ``cfg5``  B=16, H_q=32, H_kv=8, d=128, T=16384; K, V N(0,1) bf16; queries and 4096
            calibration queries per KV head: q = A_h w + eps, A_h a seeded orthonormal d x 24
            basis per KV head, w ~ N(0, I_24), eps ~ N(0, 0.01 I).
"""

from dataclasses import dataclass, field

import numpy as np

CONFIGS = {
    "cfg1": dict(B=1, Hq=1, Hkv=1, d=128, T=1024, dtype="f32", seed=0, schemes=[("tq", 4)]),
    "cfg2": dict(B=8, Hq=32, Hkv=8, d=128, T=32768, dtype="bf16", seed=1,
                 schemes=[("plain", 4), ("tq", 4), ("kqv", 4), ("qkqv", 4)]),
    "cfg3": dict(B=4, Hq=8, Hkv=8, d=1024, T=8192, dtype="bf16", seed=2,
                 schemes=[("tq", 2), ("tq", 4), ("kqv", 2), ("kqv", 4)]),
    "cfg4": dict(B=1, Hq=64, Hkv=8, d=128, T=131072, dtype="bf16", seed=3,
                 schemes=[("kqv", 2), ("kqv", 3), ("kqv", 4)], append_chunk=4096),
    "cfg5": dict(B=16, Hq=32, Hkv=8, d=128, T=16384, dtype="bf16", seed=4,
                 schemes=[("headq", 2)], headq_rank=16, calib=4096),
    # SQU-KV regime: structured (rank-16) keys and values per KV head, with separate calibration
    # sets for K and V ([ABL] "Recomendações Práticas" 2), at the headline shape
    "sq": dict(B=8, Hq=32, Hkv=8, d=128, T=32768, dtype="bf16", seed=5,
               schemes=[("squ", 2), ("tq", 2)], calib=4096),
}


def bf16_bits(x):
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _orthonormal(rng, d, r):
    q, _ = np.linalg.qr(rng.standard_normal((d, r)))
    return q


@dataclass
class Inputs:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    T: int
    dtype: str           # "f32" or "bf16"
    K: np.ndarray        # [B][Hkv][T][d]: float32, or uint16 bf16 bits
    V: np.ndarray
    q: np.ndarray        # [B][Hq][d] float32
    seed: int
    extra: dict = field(default_factory=dict)

    def k_f32(self):
        return self.K if self.dtype == "f32" else bf16_to_f32(self.K)

    def v_f32(self):
        return self.V if self.dtype == "f32" else bf16_to_f32(self.V)


def make_inputs(name, B=None, T=None, Hkv=None, Hq=None, d=None, seed=None):
    """Inputs of configuration ``name``; sizes may be overridden for scaled-down cases."""
    c = dict(CONFIGS[name])
    B = c["B"] if B is None else B
    T = c["T"] if T is None else T
    Hkv = c["Hkv"] if Hkv is None else Hkv
    Hq = c["Hq"] if Hq is None else Hq
    d = c["d"] if d is None else d
    seed = c["seed"] if seed is None else seed
    rng = np.random.default_rng(seed)
    dt = c["dtype"]
    shape = (B, Hkv, T, d)
    store = np.float32 if dt == "f32" else np.uint16
    K = np.empty(shape, dtype=store)
    V = np.empty(shape, dtype=store)
    conv = (lambda a: a.astype(np.float32)) if dt == "f32" else (lambda a: bf16_bits(a))
    extra = {}

    if name == "cfg1":
        K[...] = rng.standard_normal(shape, dtype=np.float32)
        V[...] = rng.standard_normal(shape, dtype=np.float32)
        q = rng.standard_normal((B, Hq, d), dtype=np.float32)
    elif name == "cfg2":
        s = np.sqrt(3.0)
        for b in range(B):
            for h in range(Hkv):
                K[b, h] = conv(rng.standard_t(3.0, size=(T, d)) / s)
        for b in range(B):
            for h in range(Hkv):
                V[b, h] = conv(rng.standard_t(3.0, size=(T, d)) / s)
        q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    elif name == "cfg3":
        U = _orthonormal(rng, d, 16)
        for b in range(B):
            for h in range(Hkv):
                z = rng.standard_normal((T, 16))
                K[b, h] = conv(z @ U.T + 0.1 * rng.standard_normal((T, d)))
        for b in range(B):
            for h in range(Hkv):
                V[b, h] = conv(rng.standard_normal((T, d)))
        w = rng.standard_normal((B, Hq, 16))
        q = (w @ U.T + 0.1 * rng.standard_normal((B, Hq, d))).astype(np.float32)
        extra["U"] = U
    elif name == "cfg4":
        lo, hi = np.log(0.1), np.log(10.0)
        sk = np.exp(rng.uniform(lo, hi, size=(Hkv, d)))
        sv = np.exp(rng.uniform(lo, hi, size=(Hkv, d)))
        for b in range(B):
            for h in range(Hkv):
                K[b, h] = conv(sk[h] * rng.standard_normal((T, d)))
        for b in range(B):
            for h in range(Hkv):
                V[b, h] = conv(sv[h] * rng.standard_normal((T, d)))
        q = rng.standard_normal((B, Hq, d)).astype(np.float32)
        extra.update(k_std=sk, v_std=sv)
    elif name == "sq":
        # per KV head: K = z U_K^T + eps, V = w U_V^T + eps (rank 16, eps variance 0.01),
        # queries in the key subspace; 4096 calibration vectors per head and side, fresh draws
        UK = np.stack([_orthonormal(rng, d, 16) for _ in range(Hkv)])
        UV = np.stack([_orthonormal(rng, d, 16) for _ in range(Hkv)])
        for b in range(B):
            for h in range(Hkv):
                K[b, h] = conv(rng.standard_normal((T, 16)) @ UK[h].T + 0.1 * rng.standard_normal((T, d)))
        for b in range(B):
            for h in range(Hkv):
                V[b, h] = conv(rng.standard_normal((T, 16)) @ UV[h].T + 0.1 * rng.standard_normal((T, d)))
        G = Hq // Hkv
        q = np.empty((B, Hq, d), dtype=np.float32)
        for b in range(B):
            for h in range(Hq):
                q[b, h] = UK[h // G] @ rng.standard_normal(16) + 0.1 * rng.standard_normal(d)
        n_cal = c["calib"]
        calib_k = np.stack([rng.standard_normal((n_cal, 16)) @ UK[h].T + 0.1 * rng.standard_normal((n_cal, d))
                            for h in range(Hkv)])
        calib_v = np.stack([rng.standard_normal((n_cal, 16)) @ UV[h].T + 0.1 * rng.standard_normal((n_cal, d))
                            for h in range(Hkv)])
        extra.update(UK=UK, UV=UV, calib_k=calib_k, calib_v=calib_v)
    elif name == "cfg5":
        for b in range(B):
            for h in range(Hkv):
                K[b, h] = conv(rng.standard_normal((T, d)))
        for b in range(B):
            for h in range(Hkv):
                V[b, h] = conv(rng.standard_normal((T, d)))
        A = np.stack([_orthonormal(rng, d, 24) for _ in range(Hkv)])  # [Hkv][d][24]
        G = Hq // Hkv
        q = np.empty((B, Hq, d), dtype=np.float32)
        for b in range(B):
            for h in range(Hq):
                q[b, h] = A[h // G] @ rng.standard_normal(24) + 0.1 * rng.standard_normal(d)
        n_cal = c["calib"]
        calib = np.stack([rng.standard_normal((n_cal, 24)) @ A[h].T + 0.1 * rng.standard_normal((n_cal, d))
                          for h in range(Hkv)])
        extra.update(A=A, calib=calib)
    else:
        raise KeyError(name)
    return Inputs(name, B, Hq, Hkv, d, T, dt, K, V, q, seed, extra)
