"""SQU-KV (spectral keys and values, head dim 128) on the GPU against the oracle.

Calibration (oracle/spectral.py: eigenbasis of each side's calibration set, per KV head) gives
one fp32 table set.  The GPU receives it in eigen-rank order and permutes it into the storage
order; the oracle takes the same values already permuted.  The fields the GPU writes are held to
the parity rule, and the decode is compared with the oracle's decode of the GPU-written cache
and of the oracle's own cache.
"""

import numpy as np
import pytest

from gpu_helpers import ATTN_TOL, check_exempt, compare_slab, rel_err, small_inputs, to_torch
from oracle import codec as ocodec
from oracle import spectral
from oracle.pipeline import OracleContext

pytestmark = pytest.mark.gpu


def sq_tables(inp):
    out = {}
    for side, key in (("k", "calib_k"), ("v", "calib_v")):
        rank, store = [], []
        for h in range(inp.Hkv):
            E, lam, _ = spectral.calibrate(inp.extra[key][h])
            rank.append(spectral.rank_tables(E, lam))
            store.append(spectral.storage_tables(E, lam, side))
        out[side] = (rank, store)
    return out


class SqPair:
    def __init__(self, inp, cap=None):
        import torch
        from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
        self.inp = inp
        cap = cap or (inp.T + 63) // 64 * 64
        tabs = sq_tables(inp)
        self.gpu = QuantizedKVCache(inp.d, inp.Hq, inp.Hkv, inp.B, cap, scheme="squ", n=2, seed=inp.seed)
        for i, side in enumerate("kv"):
            E = torch.from_numpy(np.stack([e for e, _ in tabs[side][0]])).cuda()
            s = torch.from_numpy(np.stack([s for _, s in tabs[side][0]])).cuda()
            self.gpu.set_spectral_basis(i, E, s)
        kc, vc = ocodec.scheme_codecs("squ", 2)
        self.orc = OracleContext(inp.d, inp.Hq, inp.Hkv, inp.B, cap, kc, vc, inp.seed,
                                 spectral_k=tabs["k"][1], spectral_v=tabs["v"][1])
        self.tabs = tabs

    def append(self, chunk):
        import torch
        for s0 in range(0, self.inp.T, chunk):
            e = min(self.inp.T, s0 + chunk)
            self.gpu.append(to_torch(self.inp.K[:, :, s0:e], self.inp.dtype).cuda(),
                            to_torch(self.inp.V[:, :, s0:e], self.inp.dtype).cuda(), [s0] * self.inp.B)
        torch.cuda.synchronize()


def _check_fields(pair, T):
    buf = pair.gpu.cache.cpu().numpy()
    ex, n = 0, 0
    for b in range(pair.inp.B):
        for h in range(pair.inp.Hkv):
            e, c = compare_slab(pair, buf, b, h, T)
            ex += e
            n += c
    check_exempt(ex, n)
    return buf


@pytest.mark.parametrize("hq,hkv,lens", [(8, 2, [300, 131]), (16, 2, [1, 300]), (2, 2, [0, 77])])
def test_squ_fields_and_decode(hq, hkv, lens):
    import torch
    inp = small_inputs("sq", B=2, T=300, Hkv=hkv, Hq=hq, seed=51)
    pair = SqPair(inp)
    pair.append(chunk=77)
    buf = _check_fields(pair, inp.T)
    out = pair.gpu.decode(torch.from_numpy(inp.q).cuda(), lens).cpu().numpy().astype(np.float64)
    ref = pair.orc.decode(buf, inp.q, lens)
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(out[b] == 0)
    assert rel_err(out, ref) <= ATTN_TOL, rel_err(out, ref)
    obuf = pair.orc.new_cache()
    pair.orc.append(obuf, inp.k_f32().astype(np.float64), inp.v_f32().astype(np.float64), [0] * inp.B)
    ref2 = pair.orc.decode(obuf, inp.q, lens)
    assert rel_err(out, ref2) <= ATTN_TOL, rel_err(out, ref2)


def test_squ_dequantize_matches_reconstruction():
    inp = small_inputs("sq", B=1, T=150, Hkv=2, seed=52)
    pair = SqPair(inp)
    pair.append(chunk=150)
    buf = pair.gpu.cache.cpu().numpy()
    for h in range(inp.Hkv):
        k, v = pair.gpu.dequantize(0, h, 0, inp.T)
        Kh, Vh = pair.orc.reconstruct(buf, 0, h, inp.T)
        for got, want in ((k, Kh), (v, Vh)):
            got = got.cpu().numpy().astype(np.float64)
            assert np.max(np.abs(got - want)) <= 1e-5 * np.max(np.abs(want)), np.max(np.abs(got - want))


def test_squ_multi_query_and_paged_pool():
    import torch
    from turboquant_quantized_kv_tq_gb300 import PagedKVCache
    inp = small_inputs("sq", B=2, T=200, Hkv=2, Hq=8, seed=53)
    pair = SqPair(inp)
    pair.append(chunk=100)
    buf = pair.gpu.cache.cpu().numpy()
    rng = np.random.default_rng(54)
    qm = rng.standard_normal((inp.B, 2, inp.Hq, inp.d)).astype(np.float32)
    lens = [200, 95]
    out = pair.gpu.decode_multi(torch.from_numpy(qm).cuda(), lens).cpu().numpy().astype(np.float64)
    for i in range(2):
        seq_i = [L - 1 + i for L in lens]
        assert rel_err(out[:, i], pair.orc.decode(buf, qm[:, i], seq_i)) <= ATTN_TOL
    # the same cache as a paged pool (shuffled pages): bit-identical records, same decode
    mb = 13
    pool = PagedKVCache(inp.d, inp.Hq, inp.Hkv, inp.B, inp.B * mb + 3, mb, scheme="squ", n=2, seed=inp.seed)
    for i, side in enumerate("kv"):
        pool.set_spectral_basis(i, torch.from_numpy(np.stack([e for e, _ in pair.tabs[side][0]])).cuda(),
                                torch.from_numpy(np.stack([s for _, s in pair.tabs[side][0]])).cuda())
    table = rng.permutation(inp.B * mb + 3)[: inp.B * mb].reshape(inp.B, mb).astype(np.int32)
    tdev = torch.from_numpy(table).cuda()
    for s0 in range(0, inp.T, 100):
        pool.append(to_torch(inp.K[:, :, s0:s0 + 100], inp.dtype).cuda(),
                    to_torch(inp.V[:, :, s0:s0 + 100], inp.dtype).cuda(),
                    torch.full((inp.B,), s0, dtype=torch.int32, device="cuda"), tdev)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    outp = pool.decode(torch.from_numpy(qm).cuda(), seq, tdev).cpu().numpy().astype(np.float64)
    for i in range(2):
        seq_i = [L - 1 + i for L in lens]
        assert rel_err(outp[:, i], pair.orc.decode(buf, qm[:, i], seq_i)) <= ATTN_TOL
    praw = pool.pool.cpu().numpy()
    L = pool.layout
    for side_off, nb, foff in ((L.k_offset, L.k_block_bytes, pair.gpu.layout.k_offset),
                               (L.v_offset, L.v_block_bytes, pair.gpu.layout.v_offset)):
        for b in range(inp.B):
            for h in range(inp.Hkv):
                for j in range((inp.T + 15) // 16):
                    a = side_off + (int(table[b, j]) * inp.Hkv + h) * nb
                    c = foff + ((b * inp.Hkv + h) * (pair.gpu.capacity // 16) + j) * nb
                    assert np.array_equal(praw[a:a + nb], buf[c:c + nb]), (b, h, j)


def test_squ_needs_its_basis_and_limits():
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache, TQError
    kv = QuantizedKVCache(128, 8, 2, 1, 64, scheme="squ", n=2, seed=1)
    q = torch.zeros(1, 8, 128, device="cuda")
    with pytest.raises(TQError) as e:  # no basis yet
        kv.decode(q, [10])
    assert e.value.status == 7
    inp = small_inputs("sq", B=1, T=64, Hkv=2, Hq=8, seed=55)
    pair = SqPair(inp, cap=64)
    pair.append(chunk=64)
    with pytest.raises(TQError) as e:  # corrected logits are not built for this codec
        pair.gpu.logits(torch.from_numpy(inp.q).cuda(), [64])
    assert e.value.status == 2
