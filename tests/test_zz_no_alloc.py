"""The allocation-free decode entry point (tq_decode_attention_static).

Some callers cannot allocate device memory where they call the decode: code running inside
another framework's stream without access to its allocator, decode loops whose memory is
planned up front (a cudaMalloc may synchronize the device), plugins handed only input and
output pointers.  For them the library keeps a built-in 8 MiB device scratch.  These tests call
that entry point through the C ABI twice in a row and check each result against the regular
entry point, which takes a caller-allocated workspace (same kernels, same work split, so the
outputs are also bit-identical), read the scratch's error word back, and check a head-dim-1024
value-sketch configuration (which uses the scratch's sketch regions and the extra sketch
launches) against the oracle.  The file is collected last.
"""

import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _cache_and_inputs():
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
    from workloads import make_inputs
    inp = make_inputs("cfg2", B=2, T=700, Hkv=2, Hq=8, seed=21)
    kv = QuantizedKVCache(128, 8, 2, 2, 704, scheme="kqv", n=4, seed=21)
    k = torch.from_numpy(inp.K.view(np.int16)).view(torch.bfloat16).cuda()
    v = torch.from_numpy(inp.V.view(np.int16)).view(torch.bfloat16).cuda()
    kv.append(k, v, [0, 0])
    return kv, torch.from_numpy(inp.q).cuda()


def _static_error_word(stream):
    from turboquant_quantized_kv_tq_gb300 import binding as b
    code = ctypes.c_int32(-1)
    st = b.tq_get_static_device_error(ctypes.byref(code), stream)
    return st, code.value


def test_static_scratch_decode_matches_workspace_decode():
    import torch
    from turboquant_quantized_kv_tq_gb300 import binding as b
    kv, q = _cache_and_inputs()
    seq = [700, 555]
    ref = kv.decode(q, seq).cpu().numpy()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        b.check(b.tq_decode_attention_static(kv._ctx, kv.cache.data_ptr(), q.data_ptr(), b.int_array(seq),
                                             out.data_ptr(), stream))
        torch.cuda.synchronize()
        assert _static_error_word(stream) == (b.TQ_OK, 0)
        got = out.cpu().numpy()
        err = np.max(np.abs(got - ref), axis=-1) / np.max(np.abs(ref), axis=-1)
        assert float(np.max(err)) <= 2e-3
        assert np.array_equal(got, ref)


def test_static_scratch_wide_value_sketch_against_oracle():
    """d = 1024, KQV n = 2: the value-sketch product runs after the decode on the scratch's
    sketch regions; two calls in a row, each against the oracle's decode of the GPU cache."""
    import torch
    from tests.gpu_helpers import ATTN_TOL, Pair, rel_err, small_inputs
    from turboquant_quantized_kv_tq_gb300 import binding as b
    inp = small_inputs("cfg3", B=2, T=150, Hkv=2)
    pair = Pair(inp, "kqv", 2)
    pair.append_gpu(chunk=64)
    buf = pair.gpu_bytes()
    seq = [150, 97]
    ref = pair.orc.decode(buf, inp.q, seq)
    q = torch.from_numpy(inp.q).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    ws_out = pair.gpu.decode(q, seq).cpu().numpy()  # the same kernels and split on a workspace
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        b.check(b.tq_decode_attention_static(pair.gpu._ctx, pair.gpu.cache.data_ptr(), q.data_ptr(),
                                             b.int_array(seq), out.data_ptr(), stream))
        torch.cuda.synchronize()
        assert _static_error_word(stream) == (b.TQ_OK, 0)
        assert np.array_equal(out.cpu().numpy(), ws_out)
        got = out.cpu().numpy().astype(np.float64)
        assert rel_err(got, ref) <= ATTN_TOL, rel_err(got, ref)


def test_static_scratch_rejects_oversized_configurations():
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
    from turboquant_quantized_kv_tq_gb300 import binding as b
    # 512 x 8 slabs need 512 * 8 * 8 * 260 * 4 bytes of partials: more than the 8 MiB scratch
    kv = QuantizedKVCache(128, 64, 8, 512, 64, scheme="kqv", n=4, seed=0)
    q = torch.zeros(512, 64, 128, device="cuda")
    out = torch.zeros_like(q)
    st = b.tq_decode_attention_static(kv._ctx, kv.cache.data_ptr(), q.data_ptr(), b.int_array([1] * 512),
                                      out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == b.TQ_ERR_WORKSPACE
    assert b"built-in scratch" in b.tq_last_error()
