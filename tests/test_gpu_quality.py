"""The quality report's GPU pipeline on a tiny case: each row's metrics, computed from the
library's dequantized cache and decode output, are recomputed from the oracle's reading of the
same stored bytes (its float64 reconstruction and its decode) and must agree."""

import os
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.mark.parametrize("name,sizes,schemes", [
    ("cfg2", dict(B=1, Hkv=2, T=96), [("tq", 4), ("qkqv", 3)]),
    ("cfg3", dict(B=1, Hkv=1, T=64, score_std=3.0), [("kqv", 2)]),
])
def test_quality_rows_match_the_oracle_reading(name, sizes, schemes):
    import quality
    from oracle import codec as ocodec
    from oracle.pipeline import OracleContext
    keep = []
    rows = quality.run_regime(name, "test", sizes, schemes, "cuda:0", keep=keep)
    assert len(rows) == len(schemes) == len(keep)
    for row, (scheme, n, kv, inp, q32) in zip(rows, keep):
        B, Hq, Hkv, d, T = inp.B, inp.Hq, inp.Hkv, inp.d, inp.T
        G = Hq // Hkv
        kc, vc = ocodec.scheme_codecs(scheme, n)
        orc = OracleContext(d, Hq, Hkv, B, kv.capacity, kc, vc, inp.seed)
        buf = kv.cache.cpu().numpy()
        Kh = np.zeros((B, Hkv, T, d))
        Vh = np.zeros((B, Hkv, T, d))
        for b in range(B):
            for h in range(Hkv):
                Kh[b, h], Vh[b, h] = orc.reconstruct(buf, b, h, T)
        K = inp.k_f32().astype(np.float64)
        V = inp.v_f32().astype(np.float64)
        q = q32.astype(np.float64)
        o_ref = quality._reference_output(q, K, V, d, G)
        o_orc = orc.decode(buf, q32, [T] * B)
        ref = quality._row(name, "test", scheme, n, K, V, Kh, Vh, q, o_ref, o_orc, d, G)
        for key in ("K_relmse", "K_dir", "V_relmse", "V_dir", "kl"):
            assert row[key] == pytest.approx(ref[key], rel=1e-3, abs=1e-7), key
        for key in ("out_relmse", "out_dir"):  # the decode tolerance, on a ratio of small numbers
            assert row[key] == pytest.approx(ref[key], rel=5e-2, abs=1e-6), key
        assert abs(row["top5"] - ref["top5"]) <= 0.1
