"""The decode step (tq_append_decode_attention): the step's n_new tokens are appended as each
sequence's last ones, then q is decoded over the whole sequence, with the query preparation
running beside the append and the decode's first reads kept off the new tokens until the append
has completed.  The step must leave exactly the cache bytes, and give exactly the output, of
tq_quantize_append followed by tq_decode_attention; the oracle decodes the step's cache as in
the parity tests.

Cases: full-length and ragged sequences; sequences of one to three tiles, where every pair stage
a warp would copy early holds a new token (all of them wait); several new tokens that cross a
tile boundary; a 64-token step (the four-lane encoder and 64-vector sketch blocks); G = 8
(separate query lo terms); n_new = 0; a length below n_new (refused, cache untouched); and the
step captured in a CUDA graph and replayed.
"""

import numpy as np
import pytest

from tests.gpu_helpers import ATTN_TOL, Pair, check_exempt, compare_slab, rel_err, small_inputs, to_torch

pytestmark = pytest.mark.gpu

SCHEMES = [("plain", 4), ("tq", 4), ("kqv", 4), ("qkqv", 4), ("tq", 2), ("qkqv", 2)]


def _new_tokens(inp, lens, n_new):
    """k, v [B][H_kv][n_new][d] on the device: tokens lens[b] - n_new .. lens[b] - 1 of slab b."""
    k = np.stack([inp.K[b, :, L - n_new:L] for b, L in enumerate(lens)])
    v = np.stack([inp.V[b, :, L - n_new:L] for b, L in enumerate(lens)])
    return to_torch(k, inp.dtype).cuda(), to_torch(v, inp.dtype).cuda()


def _step_pair(inp, scheme, n, lens, n_new, chunk=64):
    """Two caches filled alike with tokens [0, T); one takes the step, the other append + decode."""
    import torch
    a, b = Pair(inp, scheme, n), Pair(inp, scheme, n)
    q = torch.from_numpy(inp.q).cuda()
    k, v = _new_tokens(inp, lens, n_new)
    for p in (a, b):
        p.append_gpu(0, inp.T, chunk=chunk)
        # the step's slots first hold the negated tokens, so a write the step misses shows
        p.gpu.append(-k, -v, [L - n_new for L in lens])
    out_step = a.gpu.append_decode(k, v, q, lens)
    b.gpu.append(k, v, [L - n_new for L in lens])
    out_ref = b.gpu.decode(q, lens)
    torch.cuda.synchronize()
    return a, b, out_step.cpu().numpy(), out_ref.cpu().numpy()


def _check(a, b, out_step, out_ref, lens):
    buf = a.gpu_bytes()
    assert np.array_equal(buf, b.gpu_bytes()), "cache bytes differ from append + decode"
    ex, nc = 0, 0
    for bb in range(a.inp.B):  # every stored token is the input's own, the step's included
        for h in range(a.inp.Hkv):
            e, c = compare_slab(a, buf, bb, h, a.inp.T)
            ex, nc = ex + e, nc + c
    check_exempt(ex, nc)
    assert np.array_equal(out_step, out_ref), np.max(np.abs(out_step - out_ref))
    ref = a.orc.decode(a.gpu_bytes(), a.inp.q, lens)
    assert rel_err(out_step.astype(np.float64), ref) <= ATTN_TOL, rel_err(out_step.astype(np.float64), ref)


@pytest.mark.parametrize("scheme,n", SCHEMES)
def test_step_full_and_ragged(scheme, n):
    inp = small_inputs("cfg2", B=3, T=301, Hkv=2)
    lens = [301, 250, 97]
    _check(*_step_pair(inp, scheme, n, lens, 1), lens)


@pytest.mark.parametrize("scheme,n", [("plain", 4), ("kqv", 4), ("qkqv", 4)])
@pytest.mark.parametrize("lens", [[1, 5], [16, 17], [33, 48]])
def test_step_every_early_copy_waits(scheme, n, lens):
    inp = small_inputs("cfg2", B=2, T=64, Hkv=2)
    _check(*_step_pair(inp, scheme, n, lens, 1), lens)


@pytest.mark.parametrize("scheme,n", [("tq", 4), ("kqv", 4), ("qkqv", 3)])
def test_step_several_tokens_across_a_tile(scheme, n):
    inp = small_inputs("cfg2", B=2, T=200, Hkv=2)
    lens = [18, 200]
    _check(*_step_pair(inp, scheme, n, lens, 3), lens)
    lens = [40, 150]
    _check(*_step_pair(inp, scheme, n, lens, 20), lens)


@pytest.mark.parametrize("scheme,n", [("tq", 4), ("kqv", 4), ("qkqv", 4)])
def test_step_large_append(scheme, n):
    # 2 x 2 x 64 = 256 vectors per side: the four-lane encoder, 64-vector sketch blocks
    inp = small_inputs("cfg2", B=2, T=300, Hkv=2)
    lens = [300, 200]
    _check(*_step_pair(inp, scheme, n, lens, 64), lens)


@pytest.mark.parametrize("n", [2, 4])
def test_step_g8(n):
    inp = small_inputs("cfg4", B=1, T=777, Hkv=2)
    lens = [777]
    _check(*_step_pair(inp, "kqv", n, lens, 1), lens)


def test_step_without_new_tokens_is_the_decode():
    import torch
    inp = small_inputs("cfg2", B=2, T=120, Hkv=2)
    a = Pair(inp, "kqv", 4)
    a.append_gpu(chunk=64)
    q = torch.from_numpy(inp.q).cuda()
    k = torch.zeros((2, 2, 0, inp.d), dtype=torch.bfloat16, device="cuda")
    before = a.gpu_bytes()
    out = a.gpu.append_decode(k, k, q, [120, 77]).cpu().numpy()
    ref = a.gpu.decode(q, [120, 77]).cpu().numpy()
    assert np.array_equal(out, ref)
    assert np.array_equal(before, a.gpu_bytes())


def test_step_refuses_a_length_below_n_new():
    import torch
    from turboquant_quantized_kv_tq_gb300 import TQError
    inp = small_inputs("cfg2", B=2, T=64, Hkv=2)
    a = Pair(inp, "tq", 4)
    a.append_gpu(chunk=64)
    before = a.gpu_bytes()
    k, v = _new_tokens(inp, [64, 64], 3)
    q = torch.from_numpy(inp.q).cuda()
    with pytest.raises(TQError):
        a.gpu.append_decode(k, v, q, [64, 2])
    torch.cuda.synchronize()
    assert np.array_equal(before, a.gpu_bytes())


@pytest.mark.parametrize("scheme,n", [("plain", 4), ("qkqv", 4)])
def test_step_in_a_graph(scheme, n):
    import torch
    inp = small_inputs("cfg2", B=2, T=301, Hkv=2)
    lens = [301, 180]
    a, b, out_step, out_ref = _step_pair(inp, scheme, n, lens, 1)
    q = torch.from_numpy(inp.q).cuda()
    k, v = _new_tokens(inp, lens, 1)
    out = torch.zeros_like(q)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        a.gpu.workspace(max(lens))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            a.gpu.append_decode(k, v, q, lens, out=out)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), out_ref)
    assert np.array_equal(a.gpu_bytes(), b.gpu_bytes())
