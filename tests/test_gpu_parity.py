"""GPU parity: the CUDA library (through the C ABI) against the float64 oracle on identical
seeded inputs.  Sizes span several 16-token tiles, several split blocks and a ragged tail."""

import numpy as np
import pytest

from tests.gpu_helpers import (ATTN_TOL, Pair, check_exempt, compare_slab, rel_err,
                               small_inputs)

pytestmark = pytest.mark.gpu

# every codec combination the scheme constructors produce, on d = 128
SCHEMES_128 = [("plain", n) for n in (1, 2, 3, 4)] + [("tq", n) for n in (1, 2, 3, 4)] + \
              [("kqv", n) for n in (2, 3, 4)] + [("qkqv", n) for n in (2, 3, 4)]

# the configurations' own (name, scheme, n)
CONFIG_CASES = [("cfg1", "tq", 4), ("cfg2", "plain", 4), ("cfg2", "tq", 4), ("cfg2", "kqv", 4),
                ("cfg2", "qkqv", 4), ("cfg3", "tq", 2), ("cfg3", "tq", 4), ("cfg3", "kqv", 2),
                ("cfg3", "kqv", 4), ("cfg4", "kqv", 2), ("cfg4", "kqv", 3), ("cfg4", "kqv", 4),
                ("cfg5", "headq", 2)]

# head dims above 128: every codec combination built for them (no key-side QJL, no HeadQ)
WIDE_CODECS = [("plain", 1), ("tq", 2), ("tq", 3), ("tq", 4), ("kqv", 2), ("kqv", 3), ("kqv", 4)]
WIDE_CASES = [(d, s, n) for d in (256, 512, 1024) for s, n in WIDE_CODECS]


def _inputs_for(name):
    if name == "cfg1":
        return small_inputs("cfg1", B=1, T=1024, Hkv=1, Hq=1)
    if name == "cfg4":
        return small_inputs("cfg4", B=1, T=777, Hkv=2)
    if name == "cfg5":
        return small_inputs("cfg5", B=2, T=333, Hkv=2)
    return small_inputs(name, B=2, T=301, Hkv=2)


def _check_all_slabs(pair, T):
    buf = pair.gpu_bytes()
    ex, n = 0, 0
    for b in range(pair.inp.B):
        for h in range(pair.inp.Hkv):
            e, c = compare_slab(pair, buf, b, h, T)
            ex += e
            n += c
    check_exempt(ex, n)
    return buf


@pytest.mark.parametrize("name,scheme,n", CONFIG_CASES)
def test_config_append_and_decode(name, scheme, n):
    inp = _inputs_for(name)
    pair = Pair(inp, scheme, n)
    pair.append_gpu(chunk=128)
    buf = _check_all_slabs(pair, inp.T)
    seq = [inp.T - 5 * b for b in range(inp.B)]
    out = pair.decode_gpu(seq)
    # (i) the oracle decodes the GPU-written cache: isolates the decode kernel
    ref = pair.orc.decode(buf, inp.q, seq)
    assert rel_err(out, ref) <= ATTN_TOL, rel_err(out, ref)
    # (ii) end to end: the oracle's own cache from the raw inputs
    obuf = pair.orc.new_cache()
    pair.orc.append(obuf, inp.k_f32()[:, :, :inp.T].astype(np.float64),
                    inp.v_f32()[:, :, :inp.T].astype(np.float64), [0] * inp.B)
    ref2 = pair.orc.decode(obuf, inp.q, seq)
    assert rel_err(out, ref2) <= ATTN_TOL, rel_err(out, ref2)


@pytest.mark.parametrize("scheme,n", SCHEMES_128)
def test_all_schemes_d128(scheme, n):
    inp = small_inputs("cfg2", B=2, T=200, Hkv=2, seed=11)
    pair = Pair(inp, scheme, n)
    pair.append_gpu(chunk=77)
    buf = _check_all_slabs(pair, inp.T)
    seq = [200, 131]
    out = pair.decode_gpu(seq)
    ref = pair.orc.decode(buf, inp.q, seq)
    assert rel_err(out, ref) <= ATTN_TOL, rel_err(out, ref)


@pytest.mark.parametrize("d,scheme,n", WIDE_CASES)
def test_wide_head_dims(d, scheme, n):
    # G = 4 query heads per KV head; ragged lengths; 64-token append chunks
    inp = small_inputs("cfg2", B=2, T=150, Hkv=2, seed=13, d=d)
    pair = Pair(inp, scheme, n)
    pair.append_gpu(chunk=64)
    buf = _check_all_slabs(pair, inp.T)
    seq = [150, 37]
    out = pair.decode_gpu(seq)
    ref = pair.orc.decode(buf, inp.q, seq)
    assert rel_err(out, ref) <= ATTN_TOL, rel_err(out, ref)


@pytest.mark.parametrize("lens", [[0, 17], [16, 0], [1, 33]])
def test_wide_sequence_length_edge_cases(lens):
    # the value-sketch pass runs over every head, including those of empty sequences
    inp = small_inputs("cfg3", B=2, T=40, Hkv=2, seed=14)
    pair = Pair(inp, "kqv", 2)
    pair.append_gpu()
    buf = pair.gpu_bytes()
    out = pair.decode_gpu(lens)
    ref = pair.orc.decode(buf, inp.q, lens)
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(out[b] == 0)
    assert rel_err(out, ref) <= ATTN_TOL


@pytest.mark.parametrize("lens", [[0, 5], [1, 16], [15, 17], [300, 0], [299, 300]])
def test_sequence_length_edge_cases(lens):
    inp = small_inputs("cfg2", B=2, T=300, Hkv=2, seed=5)
    pair = Pair(inp, "kqv", 4)
    pair.append_gpu(chunk=300)
    buf = pair.gpu_bytes()
    out = pair.decode_gpu(lens)
    ref = pair.orc.decode(buf, inp.q, lens)
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(out[b] == 0)
    assert rel_err(out, ref) <= ATTN_TOL


# Lengths whose tile count gives the decode's split a boundary allowance above zero (at least 8
# tiles per block on a 152-SM GPU), runs of empty sequences long enough that some blocks' ranges
# hold no real tile, a one-tile sequence, and slab boundaries inside block ranges.
SPLIT_LENS = [8192] + [0] * 6 + [5000, 8192, 16] + [0] * 6


@pytest.mark.parametrize("scheme,n", [("tq", 4), ("kqv", 4), ("qkqv", 3)])
def test_split_with_boundary_allowance(scheme, n):
    inp = small_inputs("cfg2", B=16, T=8192, Hkv=2, seed=11)
    pair = Pair(inp, scheme, n)
    pair.append_gpu(chunk=4096)
    buf = pair.gpu_bytes()
    out = pair.decode_gpu(SPLIT_LENS)
    ref = pair.orc.decode(buf, inp.q, SPLIT_LENS)
    for b, L in enumerate(SPLIT_LENS):
        if L == 0:
            assert np.all(out[b] == 0)
    assert rel_err(out, ref) <= ATTN_TOL, rel_err(out, ref)


def test_ragged_starts_and_full_capacity():
    inp = small_inputs("cfg2", B=3, T=128, Hkv=2, seed=6)
    pair = Pair(inp, "tq", 3, capacity=128)
    # two appends per slab with different split points; fills the capacity exactly
    import torch
    from tests.gpu_helpers import to_torch
    for s, e in ((0, 40), (40, 128)):
        k = to_torch(inp.K[:, :, s:e], inp.dtype).cuda()
        v = to_torch(inp.V[:, :, s:e], inp.dtype).cuda()
        pair.gpu.append(k, v, [s] * 3)
    torch.cuda.synchronize()
    _check_all_slabs(pair, 128)
    with pytest.raises(Exception):
        pair.gpu.append(k, v, [100] * 3)  # 100 + 88 > capacity


def test_dequantize_matches_oracle_reconstruction():
    inp = small_inputs("cfg2", B=1, T=64, Hkv=2, seed=8)
    for scheme, n in (("kqv", 4), ("qkqv", 3), ("plain", 2)):
        pair = Pair(inp, scheme, n)
        pair.append_gpu()
        buf = pair.gpu_bytes()
        k, v = pair.gpu.dequantize(0, 1, 3, 60)
        Kr, Vr = pair.orc.reconstruct(buf, 0, 1, 60)
        for got, want in ((k, Kr[3:]), (v, Vr[3:])):
            got = got.cpu().numpy().astype(np.float64)
            assert np.max(np.abs(got - want)) <= 1e-5 * np.max(np.abs(want)) + 1e-6


def test_headq_dequantize_and_logits():
    inp = small_inputs("cfg5", B=2, T=150, Hkv=2)
    pair = Pair(inp, "headq", 2)
    pair.append_gpu()
    buf = pair.gpu_bytes()
    k, _ = pair.gpu.dequantize(1, 0, 0, 150)
    Kr, _ = pair.orc.reconstruct(buf, 1, 0, 150)
    assert np.max(np.abs(k.cpu().numpy() - Kr)) <= 1e-5 * np.max(np.abs(Kr)) + 1e-6
    import torch
    seq = [150, 97]
    lg = pair.gpu.logits(torch.from_numpy(inp.q).cuda(), seq, stride=160).cpu().numpy()
    ref = pair.orc.logits(buf, inp.q, seq, 160)
    for b, L in enumerate(seq):
        d = np.abs(lg[b, :, :L] - ref[b, :, :L])
        assert np.max(d) <= 2e-3 * np.max(np.abs(ref[b, :, :L])), np.max(d)
        assert np.all(lg[b, :, L:] == 0)


@pytest.mark.parametrize("scheme,n", [("qkqv", 4), ("tq", 4)])
def test_logits_other_key_codecs(scheme, n):
    import torch
    inp = small_inputs("cfg2", B=1, T=90, Hkv=2, seed=9)
    pair = Pair(inp, scheme, n)
    pair.append_gpu()
    buf = pair.gpu_bytes()
    lg = pair.gpu.logits(torch.from_numpy(inp.q).cuda(), [90]).cpu().numpy()
    ref = pair.orc.logits(buf, inp.q, [90], 90)
    assert np.max(np.abs(lg - ref)) <= 2e-3 * np.max(np.abs(ref))


def test_decode_is_deterministic():
    inp = small_inputs("cfg2", B=2, T=500, Hkv=2, seed=10)
    pair = Pair(inp, "kqv", 4)
    pair.append_gpu()
    a = pair.decode_gpu([500, 433])
    b = pair.decode_gpu([500, 433])
    assert np.array_equal(a, b)


def test_device_error_word_clear():
    inp = small_inputs("cfg2", B=1, T=32, Hkv=2, seed=12)
    pair = Pair(inp, "tq", 4)
    pair.append_gpu()
    pair.decode_gpu([32])
    st, code = pair.gpu.device_error()
    assert st == 0 and code == 0


def _multi_queries(inp, nq, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((inp.B, nq, inp.Hq, inp.d)).astype(np.float32)


@pytest.mark.parametrize("scheme,n,hq,hkv,nq,lens", [
    ("tq", 4, 8, 2, 2, [200, 131]),
    ("kqv", 4, 8, 2, 2, [200, 17]),
    ("qkqv", 4, 8, 2, 2, [199, 64]),
    ("tq", 3, 2, 2, 8, [100, 5]),      # G = 1: eight queries; queries 0..2 of batch 1 see nothing
    ("kqv", 4, 2, 2, 3, [100, 2]),     # G = 1, three queries: odd Gc takes the separate lo terms
    ("plain", 2, 4, 2, 4, [33, 200]),
    ("headq", 2, 8, 2, 2, [150, 97]),
])
def test_multi_query_decode(scheme, n, hq, hkv, nq, lens):
    import torch
    name = "cfg5" if scheme == "headq" else "cfg2"
    inp = small_inputs(name, B=2, T=200, Hkv=hkv, Hq=hq, seed=21)
    pair = Pair(inp, scheme, n)
    pair.append_gpu(chunk=100)
    buf = pair.gpu_bytes()
    qm = _multi_queries(inp, nq, 22)
    out = pair.gpu.decode_multi(torch.from_numpy(qm).cuda(), lens).cpu().numpy().astype(np.float64)
    for i in range(nq):
        seq_i = [max(0, L - nq + 1 + i) for L in lens]
        ref = pair.orc.decode(buf, qm[:, i], seq_i)
        for b, L in enumerate(seq_i):
            if L == 0:
                assert np.all(out[b, i] == 0)
        assert rel_err(out[:, i], ref) <= ATTN_TOL, (i, rel_err(out[:, i], ref))


@pytest.mark.parametrize("scheme", ["kqv", "qkqv"])
@pytest.mark.parametrize("hq,nq", [(2, 1), (4, 1), (2, 2), (4, 2), (2, 4)])
def test_qjl_value_readout_query_columns(scheme, hq, nq):
    # Gc = G nq query columns of 1, 2 and 4: the value sketch's readout rides in columns
    # Gc .. 2 Gc - 1 of the value MMA, as copies of the query columns' scores, and takes their
    # causal ends
    import torch
    inp = small_inputs("cfg2", B=2, T=180, Hkv=2, Hq=hq, seed=24)
    pair = Pair(inp, scheme, 4)
    pair.append_gpu(chunk=90)
    buf = pair.gpu_bytes()
    qm = _multi_queries(inp, nq, 25)
    lens = [180, 19]
    out = pair.gpu.decode_multi(torch.from_numpy(qm).cuda(), lens).cpu().numpy().astype(np.float64)
    for i in range(nq):
        seq_i = [L - nq + 1 + i for L in lens]
        assert rel_err(out[:, i], pair.orc.decode(buf, qm[:, i], seq_i)) <= ATTN_TOL, i


def test_multi_query_single_equals_decode_and_limits():
    import torch
    from turboquant_quantized_kv_tq_gb300 import TQError
    inp = small_inputs("cfg2", B=2, T=120, Hkv=2, Hq=8, seed=23)
    pair = Pair(inp, "kqv", 4)
    pair.append_gpu()
    q = torch.from_numpy(inp.q).cuda()
    a = pair.gpu.decode(q, [120, 77]).cpu().numpy()
    b = pair.gpu.decode_multi(q[:, None].contiguous(), [120, 77])[:, 0].cpu().numpy()
    assert np.array_equal(a, b)
    with pytest.raises(TQError) as e:  # G = 4: at most two queries per sequence
        pair.gpu.decode_multi(torch.zeros(2, 3, 8, 128, device="cuda"), [120, 77])
    assert e.value.status == 2
