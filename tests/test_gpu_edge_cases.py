"""GPU parity on the method's edge cases, through the C ABI against the oracle:

* zero K / V vectors (norm 0, every code by the tie rule, residual -C[c] with its signs and
  rho), on both sketch paths (16-vector `mma.sync` blocks for small appends, 64-vector
  `tcgen05` blocks for large ones; each re-takes near-zero products in fp32 FFMA);
* coordinates exactly on an fp32 decision threshold (Plain-KV with exact unit-norm fp32
  vectors, so y = x on both sides): a tie is a decision both sides must take the same way
  (the lower cell), so these codes are compared with no exemption;
* fp16 inputs on both append paths;
* extreme-range bf16 vectors (sums of squares that overflow or underflow fp32, huge and tiny
  coordinates in one vector): the stored fields under the parity rule;
* a run of one-token appends of every slab (the decode step's append) that crosses 16-token
  block boundaries and ends at full capacity.
"""

import numpy as np
import pytest

from oracle import codebook
from tests.edge_inputs import extreme_vectors, tie_vectors
from tests.gpu_helpers import ATTN_TOL, Pair, check_exempt, compare_slab, rel_err, small_inputs
from workloads import Inputs

pytestmark = pytest.mark.gpu

SMALL_CHUNK = 16   # 2 x 2 slabs x 16 tokens = 64 vectors per side: the 16-vector mma.sync sketch
LARGE_CHUNK = 150  # 600 vectors per side: the 64-vector tcgen05 sketch


def _all_slabs(pair, T):
    buf = pair.gpu_bytes()
    ex, n = 0, 0
    for b in range(pair.inp.B):
        for h in range(pair.inp.Hkv):
            e, c = compare_slab(pair, buf, b, h, T)
            ex += e
            n += c
    check_exempt(ex, n)
    return buf


def _same_decisions(orc, buf, obuf, b, h, T):
    """The two caches hold the same codes, sketch signs and side codes for slab (b, h)."""
    for side in ("k", "v"):
        g, o = orc.stored_fields(buf, side, b, h, T), orc.stored_fields(obuf, side, b, h, T)
        for f in ("codes", "signs", "side"):
            if f in g and not np.array_equal(g[f], o[f]):
                return False
    return True


def _decode_both_ways(pair, seq):
    """(i) the oracle decodes the GPU-written cache; (ii) end to end, the oracle's own cache.
    (ii) is held on the slabs whose stored decisions equal the oracle's: a code in the exempt
    zone that went the other way is a valid encoding, but in a context of a few tokens it moves
    the output by a cell width, far more than the decode tolerance."""
    inp = pair.inp
    buf = pair.gpu_bytes()
    out = pair.decode_gpu(seq)
    ref = pair.orc.decode(buf, inp.q, seq)
    assert rel_err(out, ref) <= ATTN_TOL, rel_err(out, ref)
    obuf = pair.orc.new_cache()
    pair.orc.append(obuf, inp.k_f32()[:, :, :inp.T].astype(np.float64),
                    inp.v_f32()[:, :, :inp.T].astype(np.float64), [0] * inp.B)
    ref2 = pair.orc.decode(obuf, inp.q, seq)
    G = inp.Hq // inp.Hkv
    same = [(b, h) for b in range(inp.B) for h in range(inp.Hkv)
            if _same_decisions(pair.orc, buf, obuf, b, h, int(seq[b]))]
    assert len(same) >= (inp.B * inp.Hkv + 1) // 2, len(same)
    rows = [(b, h * G + g) for b, h in same for g in range(G)]
    o2 = np.stack([out[b, hq] for b, hq in rows])
    r2 = np.stack([ref2[b, hq] for b, hq in rows])
    assert rel_err(o2, r2) <= ATTN_TOL, rel_err(o2, r2)


def _append_f16(pair, K16, V16, chunk):
    import torch
    T = K16.shape[2]
    for s in range(0, T, chunk):
        e = min(T, s + chunk)
        k = torch.from_numpy(np.ascontiguousarray(K16[:, :, s:e])).cuda()
        v = torch.from_numpy(np.ascontiguousarray(V16[:, :, s:e])).cuda()
        pair.gpu.append(k, v, [s] * pair.inp.B)
    torch.cuda.synchronize()


ZERO_CASES = [("plain", 4), ("tq", 4), ("tq", 2), ("kqv", 4), ("qkqv", 4), ("qkqv", 2), ("headq", 2)]


@pytest.mark.parametrize("chunk", [SMALL_CHUNK, LARGE_CHUNK])
@pytest.mark.parametrize("scheme,n", ZERO_CASES)
def test_zero_vectors(scheme, n, chunk):
    inp = small_inputs("cfg5" if scheme == "headq" else "cfg2", B=2, T=300, Hkv=2, seed=41)
    zk = [(0, 0, 0), (0, 0, 17), (0, 1, 100), (1, 1, 299), (1, 0, 150)]
    zv = [(0, 0, 1), (0, 0, 17), (1, 0, 150), (1, 1, 64)]
    for b, h, t in zk:
        inp.K[b, h, t] = 0
    for b, h, t in zv:
        inp.V[b, h, t] = 0
    pair = Pair(inp, scheme, n)
    pair.append_gpu(chunk=chunk)
    buf = _all_slabs(pair, inp.T)
    for side, lst, bits in (("k", zk, pair.kc.bits), ("v", zv, pair.vc.bits)):
        for b, h, t in lst:
            g = pair.orc.stored_fields(buf, side, b, h, inp.T)
            X = (inp.k_f32() if side == "k" else inp.v_f32())[b, h, :inp.T].astype(np.float64)
            o = pair.orc.encode_side(X, side, h)
            assert g["norm"][t] == 0
            # y = 0 sits on the middle threshold: every coordinate takes the cell just below it
            assert np.all(o["codes"][t] == (1 << (bits - 1)) - 1)
            assert np.array_equal(g["codes"][t], o["codes"][t])
            if "side" in g:
                assert g["side_scale"][t] == 0 and np.all(g["side"][t] == 0)
    _decode_both_ways(pair, [300, 251])


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_exact_threshold_ties_plain(n):
    d = 128
    _, thr = codebook.fp32_tables(d, n)
    X = tie_vectors(list(thr) + [0.0], d, positions=[0, 5, 64, 127])
    T = X.shape[0]
    rng = np.random.default_rng(40 + n)
    q = rng.standard_normal((1, 4, d)).astype(np.float32)
    inp = Inputs("ties", 1, 4, 1, d, T, "f32", X[None, None].copy(), X[::-1][None, None].copy(), q, 40 + n)
    pair = Pair(inp, "plain", n)
    pair.append_gpu(chunk=T)
    buf = pair.gpu_bytes()
    for side, Xs in (("k", X), ("v", X[::-1])):
        g = pair.orc.stored_fields(buf, side, 0, 0, T)
        o = pair.orc.encode_side(Xs.astype(np.float64), side, 0)
        assert np.all(g["norm"] == np.float32(1.0))
        assert np.array_equal(g["codes"], o["codes"]), np.argwhere(g["codes"] != o["codes"])[:5]
    # the oracle's decision at each planted tie is the lower cell: threshold k -> code k
    o = pair.orc.encode_side(X.astype(np.float64), "k", 0)
    targets = list(thr) + [0.0]
    for i, t in enumerate(targets):
        for jp, pos in enumerate([0, 5, 64, 127]):
            assert o["codes"][4 * i + jp, pos] == int(np.sum(thr < np.float32(t)))
    out = pair.decode_gpu([T])
    ref = pair.orc.decode(buf, q, [T])
    assert rel_err(out, ref) <= ATTN_TOL, rel_err(out, ref)


F16_CASES = [("tq", 4), ("plain", 3), ("kqv", 4), ("qkqv", 4), ("qkqv", 3), ("headq", 2)]


@pytest.mark.parametrize("chunk", [SMALL_CHUNK, LARGE_CHUNK])
@pytest.mark.parametrize("scheme,n", F16_CASES)
def test_fp16_inputs(scheme, n, chunk):
    base = small_inputs("cfg5" if scheme == "headq" else "cfg2", B=2, T=300, Hkv=2, seed=43)
    K16 = base.k_f32().astype(np.float16)
    V16 = base.v_f32().astype(np.float16)
    inp = Inputs(base.name + "-f16", base.B, base.Hq, base.Hkv, base.d, base.T, "f32",
                 K16.astype(np.float32), V16.astype(np.float32), base.q, base.seed, base.extra)
    pair = Pair(inp, scheme, n)
    _append_f16(pair, K16, V16, chunk)
    _all_slabs(pair, inp.T)
    _decode_both_ways(pair, [300, 173])


@pytest.mark.parametrize("chunk", [SMALL_CHUNK, LARGE_CHUNK])
@pytest.mark.parametrize("scheme,n", [("plain", 4), ("tq", 4), ("tq", 2), ("kqv", 4), ("qkqv", 4), ("qkqv", 2)])
def test_extreme_range_fields(scheme, n, chunk):
    """Norms (2 fp32 ulp), codes, signs and rho of vectors far outside the usual range.  The
    decode is not run on these: its value readout carries p * nu as an fp16 MMA operand."""
    rng = np.random.default_rng(47)
    B, Hkv, T, d = 2, 2, 300, 128
    K = extreme_vectors(rng, B * Hkv * T, d).reshape(B, Hkv, T, d)
    V = extreme_vectors(rng, B * Hkv * T, d).reshape(B, Hkv, T, d)
    q = rng.standard_normal((B, 4 * Hkv, d)).astype(np.float32)
    inp = Inputs("extreme", B, 4 * Hkv, Hkv, d, T, "bf16", K, V, q, 47)
    pair = Pair(inp, scheme, n)
    pair.append_gpu(chunk=chunk)
    buf = _all_slabs(pair, T)
    g = pair.orc.stored_fields(buf, "k", 0, 0, T)
    assert np.all(np.isfinite(g["norm"])) and np.all(g["norm"] > 0)


@pytest.mark.parametrize("scheme,n", [("plain", 4), ("tq", 4), ("kqv", 4), ("qkqv", 4), ("kqv", 2)])
def test_one_token_appends_to_full_capacity(scheme, n):
    # the decode step's append: B x H_kv = 64 one-token vectors per call, positions 10 .. 63,
    # crossing the blocks at 16, 32 and 48 and filling the cache to its capacity
    inp = small_inputs("cfg2", B=8, T=64, Hkv=8, Hq=32, seed=53)
    pair = Pair(inp, scheme, n, capacity=64)
    pair.append_gpu(0, 10)
    for t in range(10, 64):
        pair.append_gpu(t, t + 1)
    _all_slabs(pair, 64)
    _decode_both_ways(pair, [64, 63, 48, 47, 33, 17, 16, 1])
