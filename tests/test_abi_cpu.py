"""C-ABI checks that need no GPU: exported symbols, validation, host tables and layout vs the oracle.

The host tables are built by the library's own C++ code (Lloyd-Max by a continued-fraction
incomplete beta; SplitMix64 + Box-Muller) and compared with the oracle's independent float64
construction; no kernel runs here.
"""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import codebook, layout, tables

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

b = pytest.importorskip("turboquant_quantized_kv_tq_gb300.binding")


def _header_functions():
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = _header_functions()
    assert len(names) >= 15
    declared = {n for n, _, _ in b.DECLARATIONS}
    for n in names:
        assert hasattr(b.lib, n), n
        assert n in declared, n


def _cfg(d=128, hq=4, hkv=2, batch=2, cap=128, scheme="tq", n=4, seed=7, headq=0):
    c = b.tq_config()
    c.head_dim, c.num_q_heads, c.num_kv_heads, c.batch, c.capacity = d, hq, hkv, batch, cap
    c.qjl_m, c.headq_rank, c.headq_bits, c.seed = 0, headq, 4, seed
    b.check(b.tq_config_from_scheme(b.SCHEMES[scheme], n, c))
    return c


def _ctx(c):
    ctx = ctypes.c_void_p()
    b.check(b.tq_context_create(c, ctx))
    return ctx


def test_config_from_scheme():
    c = _cfg(scheme="kqv", n=4)
    assert (c.k.bits, c.k.rotate, c.k.qjl, c.v.bits, c.v.rotate, c.v.qjl) == (4, 1, 0, 3, 1, 1)
    c = _cfg(scheme="qkqv", n=3)
    assert (c.k.bits, c.k.qjl, c.v.bits, c.v.qjl) == (2, 1, 2, 1)
    c = _cfg(scheme="plain", n=2)
    assert (c.k.rotate, c.v.rotate) == (0, 0)
    assert b.tq_config_from_scheme(b.TQ_KQV, 1, c) == b.TQ_ERR_INVALID_ARG


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 100, b.TQ_ERR_INVALID_ARG),
    ("head_dim", 64, b.TQ_ERR_UNSUPPORTED),
    ("num_q_heads", 6, b.TQ_ERR_UNSUPPORTED),   # G = 3
    ("num_q_heads", 5, b.TQ_ERR_INVALID_ARG),   # not a multiple
    ("capacity", 100, b.TQ_ERR_INVALID_ARG),
    ("batch", 0, b.TQ_ERR_INVALID_ARG),
    ("batch", 513, b.TQ_ERR_INVALID_ARG),
])
def test_context_validation(field, value, status):
    c = _cfg()
    setattr(c, field, value)
    ctx = ctypes.c_void_p()
    assert b.tq_context_create(c, ctx) == status
    assert not ctx.value
    assert b.tq_last_error()


def test_calls_before_upload_are_refused():
    ctx = _ctx(_cfg())
    seq = b.int_array([4, 4])
    assert b.tq_decode_attention(ctx, None, None, seq, None, None, 0, None) == b.TQ_ERR_STATE
    b.tq_context_destroy(ctx)


def _blob(ctx):
    n = b.tq_tables_bytes(ctx)
    buf = np.zeros(n, dtype=np.uint8)
    b.check(b.tq_tables_host(ctx, buf.ctypes.data, n))
    return buf


def _offsets(d, m, kq, vq, hkv, rank):
    # mirror of the blob layout stated in tq.h (each array on a 256-byte boundary)
    off, out = 0, {}
    def take(name, nbytes):
        nonlocal off
        off = (off + 255) // 256 * 256
        out[name] = off
        off += nbytes
    for nm in ("k_c", "k_t", "v_c", "v_t"):
        take(nm, 64)
    take("k_sign", 4 * d)
    take("v_sign", 4 * d)
    if kq:
        take("S_K", 4 * m * d); take("S_K_T", 4 * m * d)
    if vq:
        take("S_V", 4 * m * d); take("S_V_T", 4 * m * d)
    if rank:
        take("U", 4 * hkv * d * rank)
    return out


@pytest.mark.parametrize("d", [128, 1024])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_host_codebook_matches_oracle(d, bits):
    c = _cfg(d=d, scheme="tq", n=bits)
    ctx = _ctx(c)
    blob = _blob(ctx)
    off = _offsets(d, d, 0, 0, 2, 0)
    L = 1 << bits
    cpp_c = blob[off["k_c"]:off["k_c"] + 64].view(np.float32)[:L]
    cpp_t = blob[off["k_t"]:off["k_t"] + 64].view(np.float32)[:L - 1]
    c64, t64 = codebook.lloyd_max(d, bits)
    assert np.max(np.abs(cpp_c.astype(np.float64) - c64)) <= 0.5 * np.spacing(np.abs(c64).astype(np.float32)).max()
    assert np.array_equal(cpp_c, c64.astype(np.float32))
    assert np.array_equal(cpp_t, t64.astype(np.float32))
    assert np.all(blob[off["k_t"]:off["k_t"] + 64].view(np.float32)[L - 1:] > 1e38)
    b.tq_context_destroy(ctx)


@pytest.mark.parametrize("seed", [0, 3, 12345])
def test_host_rotation_and_sketch_bit_exact(seed):
    d = 128
    c = _cfg(d=d, scheme="qkqv", n=4, seed=seed)
    ctx = _ctx(c)
    blob = _blob(ctx)
    off = _offsets(d, d, 1, 1, 2, 0)
    f = lambda name, n: blob[off[name]:off[name] + 4 * n].view(np.float32)
    assert np.array_equal(f("k_sign", d), tables.rotation_signs(seed, tables.STREAM_D_K, d).astype(np.float32))
    assert np.array_equal(f("v_sign", d), tables.rotation_signs(seed, tables.STREAM_D_V, d).astype(np.float32))
    SK = tables.sketch_matrix(seed, tables.STREAM_S_K, d, d)
    SV = tables.sketch_matrix(seed, tables.STREAM_S_V, d, d)
    assert np.array_equal(f("S_K", d * d).reshape(d, d), SK)
    assert np.array_equal(f("S_K_T", d * d).reshape(d, d), SK.T)
    assert np.array_equal(f("S_V", d * d).reshape(d, d), SV)
    assert np.array_equal(f("S_V_T", d * d).reshape(d, d), SV.T)
    assert b.tq_tables_bytes(ctx) >= off["S_V_T"] + 4 * d * d
    # the fp16 hi / lo terms of S_K then S_V for the tensor-core sketch, 8 x 8 core matrices:
    # element (i, j) at byte (i / 8) 2048 + (j / 8) 128 + (i % 8) 16 + (j % 8) 2 of each table
    start = (off["S_V_T"] + 4 * d * d + 255) // 256 * 256
    ii, jj = np.meshgrid(np.arange(128), np.arange(128), indexing="ij")
    pos = ((ii >> 3) * 2048 + (jj >> 3) * 128 + (ii & 7) * 16 + (jj & 7) * 2) // 2
    for k, S in enumerate((SK, SV)):
        o = start + k * 65536
        h16 = blob[o:o + 65536].view(np.float16).reshape(2, 128 * 128)
        hi = S.astype(np.float16)
        lo = (S - hi.astype(np.float32)).astype(np.float16)
        assert np.array_equal(h16[0][pos], hi) and np.array_equal(h16[1][pos], lo)
    b.tq_context_destroy(ctx)


def test_plain_has_unit_signs():
    c = _cfg(scheme="plain", n=3)
    ctx = _ctx(c)
    blob = _blob(ctx)
    off = _offsets(128, 128, 0, 0, 2, 0)
    assert np.all(blob[off["k_sign"]:off["k_sign"] + 512].view(np.float32) == 1.0)
    b.tq_context_destroy(ctx)


@pytest.mark.parametrize("scheme,n,headq", [("tq", 4, 0), ("kqv", 3, 0), ("qkqv", 2, 0), ("tq", 2, 16), ("plain", 1, 0)])
def test_layout_matches_oracle(scheme, n, headq):
    c = _cfg(d=128, hq=8, hkv=2, batch=3, cap=192, scheme=scheme, n=n, headq=headq)
    ctx = _ctx(c)
    lay = b.tq_cache_layout()
    b.check(b.tq_get_cache_layout(ctx, lay))
    assert lay.layout_version == 3 and lay.tile_tokens == 16
    shape = layout.CacheShape(3, 2, 192, 128, c.k.bits, bool(c.k.qjl), c.v.bits, bool(c.v.qjl), 128, headq, 4)
    want = layout.layout(shape)
    assert lay.total_bytes == want["total"]
    assert (lay.k_offset, lay.k_block_bytes) == (want["k"]["offset"], want["k"]["block"])
    assert (lay.v_offset, lay.v_block_bytes) == (want["v"]["offset"], want["v"]["block"])
    for name in b.REGION_NAMES:
        r = getattr(lay, name)
        fields = want[name[0]]["fields"]
        if name in fields:
            assert (r.offset, r.record_bytes) == fields[name], name
        else:
            assert r.record_bytes == 0, name
    b.tq_context_destroy(ctx)


@pytest.mark.parametrize("scheme,n,pages", [("tq", 4, 1), ("kqv", 4, 37), ("qkqv", 3, 5)])
def test_paged_layout(scheme, n, pages):
    # the pool's arrays are [(num_pages + 1) * H_kv] blocks of the contiguous layout's block
    # format (one extra page takes redirected accesses); the V array starts on a 256-byte boundary
    c = _cfg(d=128, hq=8, hkv=2, batch=3, cap=192, scheme=scheme, n=n)
    ctx = _ctx(c)
    flat, lay = b.tq_cache_layout(), b.tq_cache_layout()
    b.check(b.tq_get_cache_layout(ctx, flat))
    b.check(b.tq_get_paged_cache_layout(ctx, pages, lay))
    blocks = (pages + 1) * 2
    assert (lay.k_block_bytes, lay.v_block_bytes) == (flat.k_block_bytes, flat.v_block_bytes)
    assert lay.k_offset == 0
    assert lay.v_offset == (blocks * lay.k_block_bytes + 255) // 256 * 256
    assert lay.total_bytes == lay.v_offset + blocks * lay.v_block_bytes
    for name in b.REGION_NAMES:
        assert (getattr(lay, name).offset, getattr(lay, name).record_bytes) == \
            (getattr(flat, name).offset, getattr(flat, name).record_bytes), name
    assert b.tq_get_paged_cache_layout(ctx, 0, lay) == b.TQ_ERR_INVALID_ARG
    b.tq_context_destroy(ctx)


@pytest.mark.parametrize("d", [256, 1024])
def test_value_sketch_output_domain_table(d):
    # head dims above 128 with a QJL value side carry S_V R_V after the other arrays
    from oracle import rotation
    c = _cfg(d=d, scheme="kqv", n=4, seed=5)
    ctx = _ctx(c)
    blob = _blob(ctx)
    off = _offsets(d, d, 0, 1, 2, 0)
    start = (off["S_V_T"] + 4 * d * d + 255) // 256 * 256
    assert b.tq_tables_bytes(ctx) >= start + 4 * d * d
    T = blob[start:start + 4 * d * d].view(np.float32).reshape(d, d).astype(np.float64)
    SV = tables.sketch_matrix(5, tables.STREAM_S_V, d, d).astype(np.float64)
    R = rotation.rotation_matrix(tables.rotation_signs(5, tables.STREAM_D_V, d))
    want = SV @ R  # R_V^T S_V^T x = (S_V R_V)^T x
    ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(T - want) <= ulp)
    b.tq_context_destroy(ctx)


def test_spectral_scheme_config_and_validation():
    c = _cfg(scheme="squ", n=2)
    assert (c.k.bits, c.k.rotate, c.k.qjl, c.v.bits, c.v.rotate, c.v.qjl) == (2, 2, 0, 2, 2, 0)
    assert b.tq_config_from_scheme(b.TQ_SQU_KV, 3, c) == b.TQ_ERR_UNSUPPORTED
    bad = []
    c1 = _cfg(scheme="squ", n=2); c1.v.rotate = 1; bad.append(c1)        # one side only
    c2 = _cfg(scheme="squ", n=2); c2.k.bits = 3; bad.append(c2)          # not the 2-bit budget
    c3 = _cfg(scheme="squ", n=2, d=256); bad.append(c3)                  # head dim 128 only
    c4 = _cfg(scheme="squ", n=2); c4.headq_rank = 16; bad.append(c4)     # no HeadQ with it
    for c in bad:
        ctx = ctypes.c_void_p()
        assert b.tq_context_create(c, ctx) == b.TQ_ERR_UNSUPPORTED
        assert not ctx.value


def test_spectral_codebook_slots_and_layout():
    # the centroid / threshold slots of a spectral side hold the 4-bit codebook; the record is
    # the 2-bit budget (32 bytes at d = 128)
    c = _cfg(scheme="squ", n=2)
    ctx = _ctx(c)
    blob = _blob(ctx)
    c4, t4 = codebook.fp32_tables(128, 4)
    off = _offsets(128, 128, 0, 0, 4, 0)
    assert np.array_equal(blob[off["k_c"]:off["k_c"] + 64].view(np.float32), c4)
    assert np.array_equal(blob[off["k_t"]:off["k_t"] + 60].view(np.float32), t4)
    lay = b.tq_cache_layout()
    b.check(b.tq_get_cache_layout(ctx, lay))
    assert lay.k_codes.record_bytes == 32 and lay.v_codes.record_bytes == 32
    shape = layout.CacheShape(2, 2, 128, 128, 2, False, 2, False, 128, 0, 4, True, True)
    assert lay.total_bytes == layout.layout(shape)["total"]
    b.tq_context_destroy(ctx)
