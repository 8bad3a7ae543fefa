"""Paged pool with device-resident positions and lengths (tq_quantize_append_paged,
tq_decode_attention_paged) against the oracle.

The pool's pages are gathered on the host, by the layout documented in include/tq.h, into the
contiguous [B][H_kv][capacity] layout; the oracle then checks the stored fields under the parity
rule and decodes them.  Pages are handed out in a shuffled order, so logically adjacent blocks
are never adjacent in the pool.
"""

import types

import numpy as np
import pytest

from gpu_helpers import ATTN_TOL, check_exempt, compare_slab, rel_err, scheme_codecs, small_inputs, to_torch
from oracle import layout as olayout
from oracle.pipeline import OracleContext

pytestmark = pytest.mark.gpu

DEVERR_BAD_PAGE = 3
DEVERR_BAD_LENGTH = 4
TQ_ERR_DEVICE = 6  # tq_get_device_error's status when the word is set


class PagedPair:
    """A paged GPU pool, its block table, and an oracle context with capacity 16 * max_blocks."""

    def __init__(self, inp, scheme, n, max_blocks, spare_pages=5, seed=0):
        import torch
        from turboquant_quantized_kv_tq_gb300 import PagedKVCache
        self.inp = inp
        kc, vc = scheme_codecs(scheme, n)
        self.max_blocks = max_blocks
        self.num_pages = inp.B * max_blocks + spare_pages
        rng = np.random.default_rng(seed)
        pages = rng.permutation(self.num_pages)[: inp.B * max_blocks]
        self.table = pages.reshape(inp.B, max_blocks).astype(np.int32)
        self.gpu = PagedKVCache(inp.d, inp.Hq, inp.Hkv, inp.B, self.num_pages, max_blocks, scheme=None,
                                seed=inp.seed, k_codec=(kc.bits, int(kc.rotate), int(kc.qjl)),
                                v_codec=(vc.bits, int(vc.rotate), int(vc.qjl)))
        self.table_dev = torch.from_numpy(self.table).cuda()
        self.orc = OracleContext(inp.d, inp.Hq, inp.Hkv, inp.B, 16 * max_blocks, kc, vc, inp.seed)

    def append(self, t0, t1, starts=None):
        import torch
        k = to_torch(self.inp.K[:, :, t0:t1], self.inp.dtype).cuda()
        v = to_torch(self.inp.V[:, :, t0:t1], self.inp.dtype).cuda()
        st = torch.tensor([t0] * self.inp.B if starts is None else starts, dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.gpu.append(k, v, st, self.table_dev, error=err)
        torch.cuda.synchronize()
        return int(err.item())

    def gathered(self):
        """The pool's pages rearranged into the contiguous layout of the oracle's context."""
        pool = self.gpu.pool.cpu().numpy()
        lay = olayout.layout(self.orc.shape)
        L = self.gpu.layout
        assert lay["k"]["block"] == L.k_block_bytes and lay["v"]["block"] == L.v_block_bytes
        out = self.orc.new_cache()
        H = self.inp.Hkv
        for side, off, nbytes in (("k", L.k_offset, L.k_block_bytes), ("v", L.v_offset, L.v_block_bytes)):
            for b in range(self.inp.B):
                for h in range(H):
                    for j in range(self.max_blocks):
                        src = off + (int(self.table[b, j]) * H + h) * nbytes
                        dst = lay[side]["offset"] + ((b * H + h) * self.max_blocks + j) * nbytes
                        out[dst:dst + nbytes] = pool[src:src + nbytes]
        return out

    def decode(self, q, lens):
        import torch
        seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
        out = self.gpu.decode(torch.from_numpy(q).cuda(), seq, self.table_dev)
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64)


def _check_fields(pp, T):
    buf = pp.gathered()
    ex, n = 0, 0
    for b in range(pp.inp.B):
        for h in range(pp.inp.Hkv):
            e, c = compare_slab(types.SimpleNamespace(inp=pp.inp, orc=pp.orc), buf, b, h, T)
            ex += e
            n += c
    check_exempt(ex, n)
    return buf


@pytest.mark.parametrize("scheme,n", [("tq", 4), ("kqv", 4), ("qkqv", 4), ("plain", 2), ("kqv", 2)])
def test_paged_append_and_decode(scheme, n):
    inp = small_inputs("cfg2", B=3, T=200, Hkv=2, seed=31)
    pp = PagedPair(inp, scheme, n, max_blocks=16, seed=32)
    for s in range(0, inp.T, 50):  # chunks that start inside a block
        assert pp.append(s, min(inp.T, s + 50)) == 0
    buf = _check_fields(pp, inp.T)
    lens = [200, 77, 0]
    out = pp.decode(inp.q, lens)
    ref = pp.orc.decode(buf, inp.q, lens)
    assert np.all(out[2] == 0)
    assert rel_err(out, ref) <= ATTN_TOL, rel_err(out, ref)


def test_paged_many_tiles_matches_contiguous_bitwise():
    # more 16-token tiles than SMs: the device-computed split equals the host one, so the pool and
    # the contiguous cache give identical outputs; both are checked against the oracle as well
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
    inp = small_inputs("cfg2", B=8, T=640, Hkv=2, seed=41)
    pp = PagedPair(inp, "kqv", 4, max_blocks=40, seed=42)
    assert pp.append(0, inp.T) == 0
    kc, vc = scheme_codecs("kqv", 4)
    flat = QuantizedKVCache(inp.d, inp.Hq, inp.Hkv, inp.B, 640, scheme=None, seed=inp.seed,
                            k_codec=(kc.bits, int(kc.rotate), int(kc.qjl)),
                            v_codec=(vc.bits, int(vc.rotate), int(vc.qjl)))
    flat.append(to_torch(inp.K, inp.dtype).cuda(), to_torch(inp.V, inp.dtype).cuda(), [0] * inp.B)
    lens = [640, 639, 600, 333, 320, 17, 16, 1]
    buf = pp.gathered()
    assert np.array_equal(buf, flat.cache.cpu().numpy())
    out = pp.decode(inp.q, lens)
    ref_flat = flat.decode(torch.from_numpy(inp.q).cuda(), lens).cpu().numpy().astype(np.float64)
    assert np.array_equal(out, ref_flat)
    ref = pp.orc.decode(buf, inp.q, lens)
    assert rel_err(out, ref) <= ATTN_TOL, rel_err(out, ref)


def test_paged_split_with_boundary_allowance_matches_contiguous_bitwise():
    # the lengths of the contiguous split test: the device-computed split (with its boundary
    # allowance above zero and blocks whose ranges hold no real tile) equals the host one
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
    lens = [8192] + [0] * 6 + [5000, 8192, 16] + [0] * 6
    inp = small_inputs("cfg2", B=16, T=8192, Hkv=2, seed=43)
    pp = PagedPair(inp, "kqv", 4, max_blocks=512, seed=44)
    for s in range(0, inp.T, 4096):
        assert pp.append(s, s + 4096) == 0
    kc, vc = scheme_codecs("kqv", 4)
    flat = QuantizedKVCache(inp.d, inp.Hq, inp.Hkv, inp.B, 8192, scheme=None, seed=inp.seed,
                            k_codec=(kc.bits, int(kc.rotate), int(kc.qjl)),
                            v_codec=(vc.bits, int(vc.rotate), int(vc.qjl)))
    for s in range(0, inp.T, 4096):
        flat.append(to_torch(inp.K[:, :, s:s + 4096], inp.dtype).cuda(),
                    to_torch(inp.V[:, :, s:s + 4096], inp.dtype).cuda(), [s] * inp.B)
    out = pp.decode(inp.q, lens)
    ref_flat = flat.decode(torch.from_numpy(inp.q).cuda(), lens).cpu().numpy().astype(np.float64)
    assert np.array_equal(out, ref_flat)
    ref = pp.orc.decode(pp.gathered(), inp.q, lens)
    assert rel_err(out, ref) <= ATTN_TOL, rel_err(out, ref)


def test_paged_per_sequence_starts_and_multi_query():
    # each sequence appends at its own device start; the chunk's last two positions decode at once
    import torch
    inp = small_inputs("cfg2", B=3, T=150, Hkv=2, Hq=8, seed=33)
    pp = PagedPair(inp, "kqv", 4, max_blocks=12, seed=34)
    starts = [0, 16, 41]
    assert pp.append(0, 120, starts=starts) == 0
    # oracle cache: the same tokens at the same positions
    obuf = pp.orc.new_cache()
    pp.orc.append(obuf, inp.k_f32()[:, :, :120].astype(np.float64), inp.v_f32()[:, :, :120].astype(np.float64),
                  starts)
    lens = [s + 120 for s in starts]
    rng = np.random.default_rng(35)
    qm = rng.standard_normal((inp.B, 2, inp.Hq, inp.d)).astype(np.float32)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = pp.gpu.decode(torch.from_numpy(qm).cuda(), seq, pp.table_dev).cpu().numpy().astype(np.float64)
    buf = pp.gathered()
    for i in range(2):
        seq_i = [L - 1 + i for L in lens]
        ref = pp.orc.decode(buf, qm[:, i], seq_i)  # decode kernel against the GPU-written pool
        assert rel_err(out[:, i], ref) <= ATTN_TOL, (i, rel_err(out[:, i], ref))
        ref2 = pp.orc.decode(obuf, qm[:, i], seq_i)  # end to end from the raw inputs
        assert rel_err(out[:, i], ref2) <= ATTN_TOL, (i, rel_err(out[:, i], ref2))


def test_paged_graph_replay_with_device_lengths():
    # one captured step (append one token + decode); positions and lengths change on the device
    # between replays
    import torch
    inp = small_inputs("cfg2", B=2, T=180, Hkv=2, seed=36)
    pp = PagedPair(inp, "tq", 4, max_blocks=12, seed=37)
    t_fill = 150
    assert pp.append(0, t_fill) == 0
    k_tok = torch.empty(inp.B, inp.Hkv, 1, inp.d, dtype=torch.bfloat16, device="cuda")
    v_tok = torch.empty_like(k_tok)
    start = torch.zeros(inp.B, dtype=torch.int32, device="cuda")
    seq = torch.zeros(inp.B, dtype=torch.int32, device="cuda")
    q = torch.from_numpy(inp.q).cuda()
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pp.gpu.workspace(16 * pp.max_blocks)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        pp.gpu.append(k_tok, v_tok, start, pp.table_dev, error=err)
        pp.gpu.decode(q, seq, pp.table_dev, out=out)
    for t in range(t_fill, inp.T):
        k_tok.copy_(to_torch(inp.K[:, :, t:t + 1], inp.dtype).cuda())
        v_tok.copy_(to_torch(inp.V[:, :, t:t + 1], inp.dtype).cuda())
        start.fill_(t)
        seq.copy_(torch.tensor([t + 1, t + 1 - 40], dtype=torch.int32))
        g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    buf = _check_fields(pp, inp.T)
    lens = [inp.T, inp.T - 40]
    ref = pp.orc.decode(buf, inp.q, lens)
    got = out.cpu().numpy().astype(np.float64)
    assert rel_err(got, ref) <= ATTN_TOL, rel_err(got, ref)


def test_paged_bad_entries_are_recorded_and_contained():
    # out-of-range table entries, positions and lengths: the kernels redirect the access to the
    # pool's extra page and record the code; the caller's pages stay as written
    import torch
    inp = small_inputs("cfg2", B=2, T=64, Hkv=2, seed=38)
    pp = PagedPair(inp, "tq", 4, max_blocks=4, seed=39)
    assert pp.append(0, 64) == 0
    before = pp.gpu.pool.clone()
    # an append past 16 * max_blocks
    assert pp.append(0, 16, starts=[64, 0]) == DEVERR_BAD_PAGE
    # that call also rewrote sequence 1's first block with the same tokens: compare the rest
    assert pp.append(0, 16) == 0
    # the caller's pages hold what they held (the redirected writes went to the extra page)
    now = pp.gpu.pool.cpu().numpy()
    was = before.cpu().numpy()
    L = pp.gpu.layout
    H = inp.Hkv
    for side_off, nbytes in ((L.k_offset, L.k_block_bytes), (L.v_offset, L.v_block_bytes)):
        for p in range(pp.num_pages):
            for h in range(H):
                a = side_off + (p * H + h) * nbytes
                assert np.array_equal(now[a:a + nbytes], was[a:a + nbytes]), (p, h)
    # a length past the table: clamped, recorded
    seq = torch.tensor([64 + 100, 30], dtype=torch.int32, device="cuda")
    pp.gpu.decode(torch.from_numpy(inp.q).cuda(), seq, pp.table_dev)
    st, code = pp.gpu.device_error()
    assert st == TQ_ERR_DEVICE and code == DEVERR_BAD_LENGTH
    # a table entry outside [0, num_pages) inside the decoded range
    bad = pp.table.copy()
    bad[1, 1] = pp.num_pages + 7
    pp.table_dev.copy_(torch.from_numpy(bad))
    seq = torch.tensor([64, 40], dtype=torch.int32, device="cuda")
    pp.gpu.decode(torch.from_numpy(inp.q).cuda(), seq, pp.table_dev)
    st, code = pp.gpu.device_error()
    assert st == TQ_ERR_DEVICE and code == DEVERR_BAD_PAGE
    # and a clean call clears the word
    pp.table_dev.copy_(torch.from_numpy(pp.table))
    pp.gpu.decode(torch.from_numpy(inp.q).cuda(), seq, pp.table_dev)
    assert pp.gpu.device_error() == (0, 0)


def test_paged_limits():
    import torch
    from turboquant_quantized_kv_tq_gb300 import PagedKVCache, TQError
    inp = small_inputs("cfg2", B=2, T=32, Hkv=2, seed=40)
    pp = PagedPair(inp, "tq", 4, max_blocks=2)
    with pytest.raises(ValueError):  # wrong table shape
        pp.gpu.decode(torch.from_numpy(inp.q).cuda(), torch.zeros(2, dtype=torch.int32, device="cuda"),
                      torch.zeros(2, 3, dtype=torch.int32, device="cuda"))
    with pytest.raises(TQError) as e:  # head dim 256 is not built for the pool
        PagedKVCache(256, 8, 2, 2, 8, 4, scheme="tq", n=4).decode(
            torch.zeros(2, 8, 256, device="cuda"), torch.zeros(2, dtype=torch.int32, device="cuda"),
            torch.zeros(2, 4, dtype=torch.int32, device="cuda"))
    assert e.value.status == 2
