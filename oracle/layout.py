"""Packed cache layout: byte streams, record sizes, regions (the storage contract).

[HEADQ] "Visão Geral do Algoritmo" 2 says only what the cache stores (the base
key and the side code); no page fixes a bit layout.  The layout below is the
library's own contract, restated here independently so that the oracle can
produce and parse cache buffers byte for byte:

* A b-bit code with ascending centroid index c is stored in sign-magnitude
  form: s = [c >= 2^(b-1)], k = c - 2^(b-1) if s else 2^(b-1) - 1 - c, so
  that C[c] = (+1 if s else -1) * M[k] with M[k] = C[2^(b-1) + k] ascending.
* A code record (one vector) is a concatenation of streams of power-of-two
  widths, each w-bit stream holding coordinate i (rotated order) in bits
  [w*i, w*i + w), least significant bit first inside each byte:
  b = 4: one 4-bit stream of (s << 3) | k;
  b = 3: a 2-bit stream of k, then a 1-bit stream of s;
  b = 2: one 2-bit stream of (s << 1) | k;
  b = 1: one 1-bit stream of s.
* QJL signs: a 1-bit stream over the m sketch rows, bit = 1 iff (S r)_i >= 0.
* HeadQ side code: r 4-bit two's-complement nibbles, zeta_0 in the low nibble.
* The cache is one buffer of regions, each starting on a 256-byte boundary,
  in this order (bracketed ones only when present):
  k_codes, k_norm (fp32), [k_signs, k_rho (fp16)], [k_side, k_side_scale (fp16)],
  v_codes, v_norm (fp32), [v_signs, v_rho (fp16)].
  Region ``name`` is an array [B][H_kv][capacity][record bytes]; the record of
  token t of (batch b, KV head h) is at index (b * H_kv + h) * capacity + t.
"""

from dataclasses import dataclass

import numpy as np

REGION_ALIGN = 256


@dataclass(frozen=True)
class CacheShape:
    batch: int
    num_kv_heads: int
    capacity: int
    head_dim: int
    k_bits: int
    k_qjl: bool
    v_bits: int
    v_qjl: bool
    m: int
    headq_rank: int = 0
    headq_bits: int = 4


def region_records(shape):
    """[(name, bytes per token)] in storage order."""
    d, m = shape.head_dim, shape.m
    regs = [("k_codes", d * shape.k_bits // 8), ("k_norm", 4)]
    if shape.k_qjl:
        regs += [("k_signs", m // 8), ("k_rho", 2)]
    if shape.headq_rank:
        regs += [("k_side", shape.headq_rank * shape.headq_bits // 8), ("k_side_scale", 2)]
    regs += [("v_codes", d * shape.v_bits // 8), ("v_norm", 4)]
    if shape.v_qjl:
        regs += [("v_signs", m // 8), ("v_rho", 2)]
    return regs


def regions(shape):
    """{name: (offset, bytes per token)} and the total buffer size."""
    slots = shape.batch * shape.num_kv_heads * shape.capacity
    out, off = {}, 0
    for name, rec in region_records(shape):
        off = (off + REGION_ALIGN - 1) // REGION_ALIGN * REGION_ALIGN
        out[name] = (off, rec)
        off += slots * rec
    return out, off


def to_sign_magnitude(c, bits):
    half = 1 << (bits - 1)
    c = np.asarray(c, dtype=np.int64)
    s = (c >= half).astype(np.int64)
    k = np.where(s == 1, c - half, half - 1 - c)
    return s, k


def from_sign_magnitude(s, k, bits):
    half = 1 << (bits - 1)
    return np.where(np.asarray(s) == 1, half + np.asarray(k), half - 1 - np.asarray(k))


def pack_stream(values, width):
    """Pack per-vector values (N x n, each < 2**width) LSB-first into N x (n*width/8) bytes."""
    values = np.asarray(values, dtype=np.int64)
    n_vec, n = values.shape
    nbytes = n * width // 8
    out = np.zeros((n_vec, nbytes), dtype=np.uint8)
    for i in range(n):
        bit = width * i
        out[:, bit // 8] |= ((values[:, i] & ((1 << width) - 1)) << (bit % 8)).astype(np.uint8)
    return out


def unpack_stream(data, width, n):
    data = np.asarray(data, dtype=np.uint8)
    vals = np.zeros((data.shape[0], n), dtype=np.int64)
    for i in range(n):
        bit = width * i
        vals[:, i] = (data[:, bit // 8].astype(np.int64) >> (bit % 8)) & ((1 << width) - 1)
    return vals


def pack_codes(c, bits):
    """Code records (N x d*bits/8 bytes) from ascending code indices (N x d)."""
    s, k = to_sign_magnitude(c, bits)
    if bits == 4:
        return pack_stream((s << 3) | k, 4)
    if bits == 3:
        return np.concatenate([pack_stream(k, 2), pack_stream(s, 1)], axis=1)
    if bits == 2:
        return pack_stream((s << 1) | k, 2)
    if bits == 1:
        return pack_stream(s, 1)
    raise ValueError("bits must be 1..4")


def unpack_codes(data, bits, d):
    if bits == 4:
        v = unpack_stream(data, 4, d)
        return from_sign_magnitude(v >> 3, v & 7, 4)
    if bits == 3:
        k = unpack_stream(data[:, : d // 4], 2, d)
        s = unpack_stream(data[:, d // 4:], 1, d)
        return from_sign_magnitude(s, k, 3)
    if bits == 2:
        v = unpack_stream(data, 2, d)
        return from_sign_magnitude(v >> 1, v & 1, 2)
    if bits == 1:
        return from_sign_magnitude(unpack_stream(data, 1, d), np.zeros((data.shape[0], d), np.int64), 1)
    raise ValueError("bits must be 1..4")


def pack_side(zeta):
    """HeadQ side code: two's-complement nibbles, LSB-first."""
    return pack_stream(np.asarray(zeta, dtype=np.int64) & 0xF, 4)


def unpack_side(data, r):
    v = unpack_stream(data, 4, r)
    return np.where(v >= 8, v - 16, v)


def region_view(buf, shape, name):
    """The region as a (B, H_kv, capacity, record bytes) uint8 view of the cache buffer."""
    regs, _ = regions(shape)
    off, rec = regs[name]
    n = shape.batch * shape.num_kv_heads * shape.capacity * rec
    return np.asarray(buf, dtype=np.uint8)[off:off + n].reshape(
        shape.batch, shape.num_kv_heads, shape.capacity, rec)


def write_fields(buf, shape, b, h, t0, fields):
    """Store encoded fields of tokens t0.. of slab (b, h) into the cache buffer (in place).

    ``fields`` maps region names to per-token records already packed as bytes
    (N x record bytes) or to scalar arrays (norms fp32, rho / scales fp16).
    """
    for name, val in fields.items():
        view = region_view(buf, shape, name)
        arr = np.asarray(val)
        if arr.dtype != np.uint8:
            arr = arr.view(np.uint8).reshape(arr.shape[0], -1)
        view[b, h, t0:t0 + arr.shape[0], :] = arr


def read_field(buf, shape, name, b, h, t0, t1, dtype=None):
    raw = region_view(buf, shape, name)[b, h, t0:t1, :].copy()
    if dtype is None:
        return raw
    return raw.view(dtype).reshape(t1 - t0)
