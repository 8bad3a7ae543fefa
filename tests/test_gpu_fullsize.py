"""GPU parity at the configurations' full sizes, in the launch configuration the benchmark uses:
the whole cache is written by the GPU in 4096-token chunks and decoded for every query head at
full context; sampled (batch, KV head) slabs are then checked against the oracle -- their stored
fields (bit-exact outside the exempt zone) and their attention outputs (within the attention
tolerance).  Every output of the full decode must be finite."""

import numpy as np
import pytest

from tests.gpu_helpers import (ATTN_TOL, Pair, check_exempt, compare_slab, rel_err)
from workloads import make_inputs

pytestmark = pytest.mark.gpu

FULL = [
    ("cfg2", [("plain", 4), ("tq", 4), ("kqv", 4), ("qkqv", 4)], [(0, 0), (7, 5)]),
    ("cfg4", [("kqv", 2), ("kqv", 3), ("kqv", 4)], [(0, 3)]),
    ("cfg3", [("tq", 2), ("tq", 4), ("kqv", 2), ("kqv", 4)], [(3, 7)]),
    ("cfg5", [("headq", 2)], [(15, 2)]),
]


@pytest.mark.parametrize("name,schemes,slabs", FULL, ids=[f[0] for f in FULL])
def test_full_size_sampled_parity(name, schemes, slabs):
    import torch
    inp = make_inputs(name)
    G = inp.Hq // inp.Hkv
    seq = [inp.T] * inp.B
    for scheme, n in schemes:
        pair = Pair(inp, scheme, n)
        pair.append_gpu(chunk=4096)
        buf = pair.gpu_bytes()
        ex, coords = 0, 0
        for b, h in slabs:
            e, c = compare_slab(pair, buf, b, h, inp.T)
            ex += e
            coords += c
        check_exempt(ex, coords)
        out = pair.decode_gpu(seq)
        assert np.all(np.isfinite(out)), (scheme, n)
        ref = pair.orc.decode(buf, inp.q, seq, slabs=slabs)
        for b, h in slabs:
            o, r = out[b:b + 1, h * G:(h + 1) * G], ref[b:b + 1, h * G:(h + 1) * G]
            assert rel_err(o, r) <= ATTN_TOL, (scheme, n, b, h, rel_err(o, r))
        del pair
        torch.cuda.empty_cache()
