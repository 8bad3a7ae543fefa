"""Chunked-prefill attention (tq_prefill_attention) against the oracle.

The chunk's nq queries are its last positions, already appended; query i attends to the first
L - nq + 1 + i tokens.  The oracle reconstructs each slab of the GPU-written cache once and runs
textbook attention for every query over its causal prefix; every output row is compared under
the decode tolerance.  Schemes with a QJL side run the mma.sync kernel, the others the tcgen05
one; the size, group and long-prefix cases run both.  Cases span nq = 16, 128 and 512 (several 128-row blocks, a ragged last
block), G = 1, 4 and 8, ragged sequence lengths (one shorter than the chunk, so some queries see
no token), every Plain / TQ-KV / KQV / QKQV codec family, and the one-query-column case against
tq_decode_attention_multi.
"""

import numpy as np
import pytest

from oracle.attention import decode_attention
from tests.gpu_helpers import ATTN_TOL, Pair, rel_err, small_inputs

pytestmark = pytest.mark.gpu


def _oracle_prefill(pair, buf, qm, lens):
    inp, orc = pair.inp, pair.orc
    B, nq, Hq, d = qm.shape
    G = Hq // inp.Hkv
    out = np.zeros((B, nq, Hq, d))
    for b in range(B):
        L = int(lens[b])
        for h in range(inp.Hkv):
            Kh, Vh = orc.reconstruct(buf, b, h, L)
            for i in range(nq):
                e = L - nq + 1 + i
                if e <= 0:
                    continue
                for g in range(G):
                    out[b, i, h * G + g] = decode_attention(qm[b, i, h * G + g].astype(np.float64), Kh[:e], Vh[:e])
    return out


def _run(scheme, n, nq, G, lens, T, seed, name="cfg2"):
    import torch
    Hkv = 2
    inp = small_inputs(name, B=len(lens), T=T, Hkv=Hkv, Hq=G * Hkv, seed=seed)
    pair = Pair(inp, scheme, n)
    pair.append_gpu(chunk=256)
    rng = np.random.default_rng(seed + 1)
    qm = rng.standard_normal((inp.B, nq, inp.Hq, inp.d)).astype(np.float32)
    out = pair.gpu.prefill(torch.from_numpy(qm).cuda(), lens)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    buf = pair.gpu_bytes()
    ref = _oracle_prefill(pair, buf, qm, lens)
    for b in range(inp.B):
        for i in range(nq):
            if lens[b] - nq + 1 + i <= 0:
                assert np.all(got[b, i] == 0), (b, i)
    err = rel_err(got.reshape(-1, inp.d), ref.reshape(-1, inp.d))
    assert err <= ATTN_TOL, err
    return pair, qm, got


@pytest.mark.parametrize("scheme,n", [("plain", 4), ("tq", 4), ("tq", 2), ("kqv", 4), ("kqv", 3), ("kqv", 2),
                                      ("qkqv", 4), ("qkqv", 3), ("plain", 1), ("tq", 3)])
def test_prefill_schemes_nq128(scheme, n):
    _run(scheme, n, nq=128, G=4, lens=[700, 311], T=700, seed=70)


# KQV (a QJL value side: 64-column scores, the value sketch readout) and TQ-KV (no sketch: wide scores)
@pytest.mark.parametrize("scheme", ["kqv", "tq"])
@pytest.mark.parametrize("nq,G,lens", [(16, 4, [333, 16, 9]), (512, 4, [900, 600]), (512, 1, [777, 513]),
                                       (128, 8, [640, 129])])
def test_prefill_chunk_sizes_and_groups(scheme, nq, G, lens):
    _run(scheme, 4, nq=nq, G=G, lens=lens, T=max(lens), seed=71 + nq + G)


@pytest.mark.parametrize("scheme", ["kqv", "tq"])
def test_prefill_outlier_channels_long_prefix(scheme):
    # the long-context recipe (per-channel std in [0.1, 10]) with a 2048-token prefix at n = 2
    _run(scheme, 2, nq=64, G=8, lens=[2048], T=2048, seed=75, name="cfg4")


def test_prefill_matches_multi_query_decode():
    # a chunk small enough for the multi-query decode (G nq <= 8): both paths, one answer
    import torch
    pair, qm, got = _run("qkqv", 4, nq=2, G=4, lens=[300, 77], T=300, seed=76)
    multi = pair.gpu.decode_multi(torch.from_numpy(qm).cuda(), [300, 77]).cpu().numpy().astype(np.float64)
    assert rel_err(got.reshape(-1, 128), multi.reshape(-1, 128)) <= ATTN_TOL


def test_prefill_rejects_unbuilt_configurations():
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
    from turboquant_quantized_kv_tq_gb300 import binding as b
    kv = QuantizedKVCache(256, 8, 2, 1, 64, scheme="tq", n=4, seed=0)
    q = torch.zeros(1, 4, 8, 256, device="cuda")
    out = torch.zeros_like(q)
    ws = torch.empty(max(256, kv.prefill_workspace_bytes(4)), dtype=torch.uint8, device="cuda")
    st = b.tq_prefill_attention(kv._ctx, kv.cache.data_ptr(), q.data_ptr(), 4, b.int_array([10]), out.data_ptr(),
                                ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == b.TQ_ERR_UNSUPPORTED
