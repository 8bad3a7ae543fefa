"""Bounds evidence without a sanitizer: every call writes only the bytes it owns.

The cache (or paged pool), the decode workspace, the outputs and 4 KiB on either side of each
are filled with the byte 0xA5 before the calls.  After each call the whole buffer is read back
and every byte outside the call's own fields must hold what it held before: the stored fields of
the appended tokens (positions from the oracle's independent layout) for an append; nothing in
the cache for a read; the first tq_decode_workspace_bytes of the workspace; the output rows; the
logits of stored tokens only.  A stray write anywhere else (another slab, tokens past the
sequence, padding between fields, the redirect page of a pool, past the workspace's end) fails.
"""

import ctypes

import numpy as np
import pytest

from oracle import layout as olayout
from tests.gpu_helpers import Pair, scheme_codecs, small_inputs, to_torch

pytestmark = pytest.mark.gpu

GUARD = 4096
FILL = 0xA5


class Guarded:
    """A device byte buffer of `nbytes` with GUARD canary bytes on either side."""

    def __init__(self, nbytes):
        import torch
        self.n = int(nbytes)
        self.buf = torch.full((GUARD + self.n + GUARD,), FILL, dtype=torch.uint8, device="cuda")

    def ptr(self):
        return self.buf.data_ptr() + GUARD

    def host(self):
        import torch
        torch.cuda.synchronize()
        return self.buf.cpu().numpy()

    def check(self, before, owned=None, what=""):
        """Bytes outside `owned` (a bool mask over the n inner bytes, or None) are unchanged."""
        after = self.host()
        keep = np.ones(after.size, dtype=bool)
        if owned is not None:
            keep[GUARD:GUARD + self.n] = ~owned
        bad = np.flatnonzero((after != before) & keep)
        assert bad.size == 0, (what, "stray writes at inner offsets", (bad[:8] - GUARD).tolist())
        return after


def _owned_append(shape, t0, t1):
    """Mask of the cache bytes an append of tokens [t0, t1) of every slab owns."""
    lay = olayout.layout(shape)
    mask = np.zeros(lay["total"], dtype=bool)
    t = np.arange(t0, t1)
    for side in ("k", "v"):
        for name in lay[side]["fields"]:
            for b in range(shape.batch):
                for h in range(shape.num_kv_heads):
                    mask[olayout.field_positions(shape, name, b, h, t)] = True
    return mask


@pytest.mark.parametrize("scheme,n,d", [("kqv", 4, 128), ("qkqv", 3, 128), ("headq", 2, 128),
                                        ("plain", 2, 128), ("kqv", 4, 1024), ("tq", 3, 256)])
def test_contiguous_calls_write_only_their_bytes(scheme, n, d):
    import torch
    from turboquant_quantized_kv_tq_gb300 import binding as b
    inp = small_inputs("cfg5" if scheme == "headq" else "cfg2", B=2, T=300, Hkv=2, seed=61, d=d)
    pair = Pair(inp, scheme, n, capacity=320)
    kv, shape = pair.gpu, pair.orc.shape
    total = int(kv.layout.total_bytes)
    assert total == olayout.layout(shape)["total"]
    cache = Guarded(total)
    st = torch.cuda.current_stream().cuda_stream
    ctx = kv._ctx
    dt = b.TQ_BF16
    before = cache.host()
    for t0, t1 in ((0, 37), (37, 300)):  # FFMA-path then tensor-core-path appends
        k = to_torch(inp.K[:, :, t0:t1], inp.dtype).cuda()
        v = to_torch(inp.V[:, :, t0:t1], inp.dtype).cuda()
        b.check(b.tq_quantize_append(ctx, cache.ptr(), k.data_ptr(), v.data_ptr(), dt, t1 - t0,
                                     b.int_array([t0] * inp.B), st))
        before = cache.check(before, _owned_append(shape, t0, t1), f"append {t0}..{t1}")

    seq = [300, 211]
    need = int(b.tq_decode_workspace_bytes(ctx, max(seq)))
    ws = Guarded(need)
    q = torch.from_numpy(inp.q).cuda()
    out = Guarded(q.numel() * 4)
    ws_before, out_before = ws.host(), out.host()
    b.check(b.tq_decode_attention(ctx, cache.ptr(), q.data_ptr(), b.int_array(seq), out.ptr(), ws.ptr(), need, st))
    cache.check(before, None, "decode: cache")
    ws_before = ws.check(ws_before, np.ones(need, dtype=bool), "decode: workspace")
    owned_out = np.ones(q.numel() * 4, dtype=bool)
    out_before = out.check(out_before, owned_out, "decode: output")
    got = out.host()[GUARD:GUARD + q.numel() * 4].view(np.float32)
    assert np.all(np.isfinite(got))

    G = inp.Hq // inp.Hkv
    if d == 128 and 2 * G <= 8:
        nq = 2
        qm = torch.from_numpy(np.random.default_rng(62).standard_normal((inp.B, nq, inp.Hq, d)).astype(np.float32)).cuda()
        outm = Guarded(qm.numel() * 4)
        om_before = outm.host()
        b.check(b.tq_decode_attention_multi(ctx, cache.ptr(), qm.data_ptr(), nq, b.int_array(seq), outm.ptr(),
                                            ws.ptr(), need, st))
        cache.check(before, None, "multi-query decode: cache")
        ws.check(ws_before, np.ones(need, dtype=bool), "multi-query decode: workspace")
        outm.check(om_before, np.ones(qm.numel() * 4, dtype=bool), "multi-query decode: output")

    if d == 128:  # corrected logits are built for head dim 128
        stride = 320
        lg = Guarded(inp.B * inp.Hq * stride * 4)
        lg_before = lg.host()
        b.check(b.tq_headq_correct(ctx, cache.ptr(), q.data_ptr(), b.int_array(seq), lg.ptr(), stride, st))
        owned = np.zeros((inp.B, inp.Hq, stride, 4), dtype=bool)
        for bb in range(inp.B):
            owned[bb, :, :seq[bb]] = True
        lg.check(lg_before, owned.ravel(), "logits")
        cache.check(before, None, "logits: cache")

    t0, t1 = 5, 77
    ko, vo = Guarded((t1 - t0) * d * 4), Guarded((t1 - t0) * d * 4)
    ko_before, vo_before = ko.host(), vo.host()
    b.check(b.tq_dequantize(ctx, cache.ptr(), 1, 0, t0, t1, ko.ptr(), vo.ptr(), st))
    ko.check(ko_before, np.ones((t1 - t0) * d * 4, dtype=bool), "dequantize k")
    vo.check(vo_before, np.ones((t1 - t0) * d * 4, dtype=bool), "dequantize v")
    cache.check(before, None, "dequantize: cache")


def _owned_paged(shape, L, table, H, t0s, n_new):
    """Mask of the pool bytes a paged append owns: each token's fields in its page's blocks."""
    lay = olayout.layout(shape)
    max_blocks = table.shape[1]
    mask = np.zeros(int(L.total_bytes), dtype=bool)
    for side, off, nbytes in (("k", L.k_offset, L.k_block_bytes), ("v", L.v_offset, L.v_block_bytes)):
        for name in lay[side]["fields"]:
            for bb in range(table.shape[0]):
                t = np.arange(t0s[bb], t0s[bb] + n_new)
                for h in range(H):
                    pos = olayout.field_positions(shape, name, bb, h, t)  # contiguous layout
                    rel = pos - lay[side]["offset"]
                    blk, inner = rel // nbytes, rel % nbytes
                    j = blk % max_blocks  # slab-major blocks: (b * H + h) * max_blocks + j
                    page = table[bb][j]
                    mask[off + (page * H + h) * nbytes + inner] = True
    return mask


@pytest.mark.parametrize("scheme,n", [("tq", 4), ("kqv", 4), ("qkqv", 2)])
def test_paged_calls_write_only_their_bytes(scheme, n):
    import torch
    from turboquant_quantized_kv_tq_gb300 import PagedKVCache
    from turboquant_quantized_kv_tq_gb300 import binding as b
    from oracle.pipeline import OracleContext
    inp = small_inputs("cfg2", B=3, T=200, Hkv=2, seed=63)
    kc, vc = scheme_codecs(scheme, n)
    max_blocks, num_pages = 14, 3 * 14 + 4
    rng = np.random.default_rng(64)
    table = rng.permutation(num_pages)[:3 * max_blocks].reshape(3, max_blocks).astype(np.int32)
    pc = PagedKVCache(128, inp.Hq, inp.Hkv, inp.B, num_pages, max_blocks, scheme=None, seed=inp.seed,
                      k_codec=(kc.bits, int(kc.rotate), int(kc.qjl)), v_codec=(vc.bits, int(vc.rotate), int(vc.qjl)))
    orc = OracleContext(128, inp.Hq, inp.Hkv, inp.B, 16 * max_blocks, kc, vc, inp.seed)
    L = pc.layout
    pool = Guarded(int(L.total_bytes))
    st = torch.cuda.current_stream().cuda_stream
    table_dev = torch.from_numpy(table).cuda()
    pt = b.tq_page_table(table_dev.data_ptr(), max_blocks, num_pages)
    before = pool.host()
    starts = [0, 9, 30]
    for t0, t1 in ((0, 21), (21, 150)):
        k = to_torch(inp.K[:, :, t0:t1], inp.dtype).cuda()
        v = to_torch(inp.V[:, :, t0:t1], inp.dtype).cuda()
        s = [x + t0 for x in starts]
        sdev = torch.tensor(s, dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        b.check(b.tq_quantize_append_paged(pc._ctx, pool.ptr(), ctypes.byref(pt), k.data_ptr(), v.data_ptr(),
                                           b.TQ_BF16, t1 - t0, sdev.data_ptr(), err.data_ptr(), st))
        before = pool.check(before, _owned_paged(orc.shape, L, table, inp.Hkv, s, t1 - t0), f"paged append {t0}..{t1}")
        assert int(err.item()) == 0
    lens = torch.tensor([x + 150 for x in starts], dtype=torch.int32, device="cuda")
    need = int(b.tq_decode_workspace_bytes(pc._ctx, 16 * max_blocks))
    ws = Guarded(need)
    q = torch.from_numpy(inp.q).cuda()
    out = Guarded(q.numel() * 4)
    ws_before, out_before = ws.host(), out.host()
    b.check(b.tq_decode_attention_paged(pc._ctx, pool.ptr(), ctypes.byref(pt), q.data_ptr(), 1, lens.data_ptr(),
                                        out.ptr(), ws.ptr(), need, st))
    pool.check(before, None, "paged decode: pool")
    ws.check(ws_before, np.ones(need, dtype=bool), "paged decode: workspace")
    out.check(out_before, np.ones(q.numel() * 4, dtype=bool), "paged decode: output")
