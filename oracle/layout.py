"""Packed cache layout: byte streams, record sizes, 16-token blocks (the storage contract).

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
* The cache holds two arrays of 16-token blocks, K then V (the V array starts
  on a 256-byte boundary).  Each array is [B][H_kv][capacity / 16] blocks; a
  block stores, for its 16 tokens, one field after another (bracketed ones only
  when present), each field 16 records long:
  K block: codes, norm (fp32), [signs, rho (fp16)], [side, side_scale (fp16)];
  V block: codes, norm (fp32), [signs, rho (fp16)].
  Token t of (batch b, KV head h) is in block
  side_offset + ((b * H_kv + h) * capacity / 16 + t // 16) * block_bytes, at
  position p = t % 16.  A field of fixed-size records stores record p at
  field_offset + p * record_bytes, except the value side's streams: the codes
  (each stream of a b = 3 code on its own, one after the other) and the QJL
  signs of a V block are stored by groups of 16 coordinates.  In a w-bit
  stream each group holds the 2w bytes of coordinates [16 g, 16 g + 16) of the
  16 tokens, [groups][16 tokens][2w bytes], so byte j of token p's record is at
  stream_offset + (j // 2w) * 32 w + p * 2w + j % 2w.  (A decoder that reads
  one coordinate group for several tokens then makes one contiguous load.)
"""

from dataclasses import dataclass

import numpy as np

TILE = 16          # tokens per block
SIDE_ALIGN = 256


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
    k_sq: bool = False  # SQU-KV sides (oracle/spectral.py): d/4-byte code records
    v_sq: bool = False


def side_fields(shape, side):
    """[(field name, bytes per token)] of one side's block, in block order."""
    d, m = shape.head_dim, shape.m
    if side == "k":
        f = [("k_codes", d // 4 if shape.k_sq else d * shape.k_bits // 8), ("k_norm", 4)]
        if shape.k_qjl:
            f += [("k_signs", m // 8), ("k_rho", 2)]
        if shape.headq_rank:
            f += [("k_side", shape.headq_rank * shape.headq_bits // 8), ("k_side_scale", 2)]
        return f
    f = [("v_codes", d // 4 if shape.v_sq else d * shape.v_bits // 8), ("v_norm", 4)]
    if shape.v_qjl:
        f += [("v_signs", m // 8), ("v_rho", 2)]
    return f


def layout(shape):
    """{side: {"offset", "block", "fields": {name: (offset in block, bytes per token)}}, "total"}."""
    assert shape.capacity % TILE == 0
    blocks = shape.batch * shape.num_kv_heads * (shape.capacity // TILE)
    out, off = {}, 0
    for side in ("k", "v"):
        off = (off + SIDE_ALIGN - 1) // SIDE_ALIGN * SIDE_ALIGN
        fields, foff = {}, 0
        for name, rec in side_fields(shape, side):
            fields[name] = (foff, rec)
            foff += TILE * rec
        out[side] = {"offset": off, "block": foff, "fields": fields}
        off += blocks * foff
    out["total"] = off
    return out


def grouped_streams(shape, name):
    """[(width w, coordinates n)] of a value-side field stored by coordinate groups, else None."""
    if name == "v_codes" and shape.v_sq:  # magnitudes then signs, 2 bytes per group each
        return [(1, shape.head_dim), (1, shape.head_dim)]
    if name == "v_codes":
        d, b = shape.head_dim, shape.v_bits
        return {4: [(4, d)], 3: [(2, d), (1, d)], 2: [(2, d)], 1: [(1, d)]}[b]
    if name == "v_signs":
        return [(1, shape.m)]
    return None


def record_byte_positions(shape, name, p):
    """In-field byte offset of each byte of the records of block positions p (array): shape
    (len(p), record bytes)."""
    p = np.asarray(p, dtype=np.int64)
    rec = dict(side_fields(shape, name[0]))[name]
    streams = grouped_streams(shape, name)
    if streams is None:
        return p[:, None] * rec + np.arange(rec)[None, :]
    cols, base = [], 0
    for w, n in streams:
        j = np.arange(n * w // 8)
        cols.append(base + (j // (2 * w))[None, :] * 32 * w + p[:, None] * 2 * w + (j % (2 * w))[None, :])
        base += TILE * n * w // 8
    return np.concatenate(cols, axis=1)


def field_positions(shape, name, b, h, t):
    """Absolute byte positions (len(t) x record bytes) of field ``name`` of tokens t of slab (b, h)."""
    lay = layout(shape)
    side = lay[name[0]]
    foff, rec = side["fields"][name]
    t = np.asarray(t, dtype=np.int64)
    slab = b * shape.num_kv_heads + h
    blk = slab * (shape.capacity // TILE) + t // TILE
    start = side["offset"] + blk * side["block"] + foff
    return start[:, None] + record_byte_positions(shape, name, t % TILE)


def field_offsets(shape, name, b, h, t):
    """Byte offset of field ``name`` of tokens t (array) of slab (b, h), for the fields stored
    as whole records (every field but the value side's streams)."""
    assert grouped_streams(shape, name) is None
    lay = layout(shape)
    side = lay[name[0]]
    foff, rec = side["fields"][name]
    t = np.asarray(t, dtype=np.int64)
    slab = b * shape.num_kv_heads + h
    blk = slab * (shape.capacity // TILE) + t // TILE
    return side["offset"] + blk * side["block"] + foff + (t % TILE) * rec, rec


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


def write_fields(buf, shape, b, h, t0, fields):
    """Store encoded fields of tokens t0.. of slab (b, h) into the cache buffer (in place).

    ``fields`` maps field names to per-token records already packed as bytes
    (N x record bytes) or to scalar arrays (norms fp32, rho / scales fp16).
    """
    buf = np.asarray(buf, dtype=np.uint8)
    for name, val in fields.items():
        arr = np.asarray(val)
        if arr.dtype != np.uint8:
            arr = arr.view(np.uint8).reshape(arr.shape[0], -1)
        buf[field_positions(shape, name, b, h, np.arange(t0, t0 + arr.shape[0]))] = arr


def read_field(buf, shape, name, b, h, t0, t1, dtype=None):
    raw = np.asarray(buf, dtype=np.uint8)[field_positions(shape, name, b, h, np.arange(t0, t1))].copy()
    if dtype is None:
        return raw
    return raw.view(dtype).reshape(t1 - t0)
