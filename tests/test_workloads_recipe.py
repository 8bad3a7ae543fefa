"""The seeded input generators (workloads.py at the repository root) against their stated
recipe, at reduced sizes: distributions, structure (rank, subspaces, per-channel scales), the bf16
rounding, shapes and seeding.  Statistical checks use bounds many standard errors wide."""

import numpy as np
import pytest

from workloads import CONFIGS, bf16_bits, bf16_to_f32, make_inputs


def _svals(X):
    return np.linalg.svd(np.asarray(X, dtype=np.float64), compute_uv=False)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, -2.5, 3.0e38, 1e-40, 0.0], dtype=np.float32)
    got = bf16_to_f32(bf16_bits(x))
    # ties go to the even mantissa: 1 + 2^-8 -> 1, 1 + 3 * 2^-8 -> 1 + 2^-6; others exact or nearest
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == np.float32(1.0 + 2.0**-6)
    assert got[3] == -2.5
    rng = np.random.default_rng(0)
    y = rng.standard_normal(10000).astype(np.float32) * 100
    yb = bf16_to_f32(bf16_bits(y)).astype(np.float64)
    assert np.all(np.abs(yb - y) <= np.abs(y) * 2.0**-8 + 1e-45)  # half an ulp of an 8-bit mantissa


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_shapes_dtypes_and_seeding(name):
    G = CONFIGS[name]["Hq"] // CONFIGS[name]["Hkv"]
    kw = dict(B=2, T=64, Hkv=2, Hq=2 * G)
    if name == "cfg1":
        kw = dict(B=1, T=64, Hkv=1, Hq=1)
    a = make_inputs(name, **kw)
    b = make_inputs(name, **kw)
    c = make_inputs(name, seed=CONFIGS[name]["seed"] + 100, **kw)
    assert a.K.shape == (a.B, a.Hkv, a.T, a.d) and a.q.shape == (a.B, a.Hkv * G, a.d)
    assert a.K.dtype == (np.float32 if CONFIGS[name]["dtype"] == "f32" else np.uint16)
    assert a.q.dtype == np.float32
    assert np.array_equal(a.K, b.K) and np.array_equal(a.V, b.V) and np.array_equal(a.q, b.q)
    assert not np.array_equal(a.K, c.K)


def test_cfg1_standard_normal():
    x = make_inputs("cfg1", T=4096)
    for t in (x.K, x.V):
        assert abs(float(t.mean())) < 0.01 and abs(float(t.var()) - 1.0) < 0.02


def test_cfg2_unit_variance_heavy_tails():
    from scipy import stats
    x = make_inputs("cfg2", B=1, Hkv=2, Hq=8, T=8192)
    for t in (x.k_f32(), x.v_f32()):
        k = t.astype(np.float64).ravel()
        # Student-t(3) / sqrt(3).  The threshold sits midway between two bf16 values (3 and
        # 3 + 2^-6), so rounding moves no sample across it: the bf16 tail is the exact one
        thr = 3.0 + 2.0**-7
        p = 2.0 * stats.t.sf(thr * np.sqrt(3.0), 3)  # 0.0137, against 0.0027 for a unit Gaussian
        se = np.sqrt(p * (1 - p) / k.size)
        assert abs(float(np.mean(np.abs(k) > thr)) - p) < 6 * se
        med = stats.t.ppf(0.75, 3) / np.sqrt(3.0)  # median of |X|
        assert abs(np.median(np.abs(k)) - med) < 0.005
    q = x.q.astype(np.float64)
    assert abs(q.mean()) < 0.1 and abs(q.var() - 1.0) < 0.1


def test_cfg3_low_rank_keys_and_queries():
    x = make_inputs("cfg3", B=1, Hkv=1, Hq=1, T=2048, d=256)
    s = _svals(x.k_f32()[0, 0])
    # 16 directions of variance 1 (singular values ~ sqrt(T)), the rest noise of variance 0.01
    assert s[15] > 0.6 * np.sqrt(2048) and s[16] < 0.2 * np.sqrt(2048)
    U = x.extra["U"]
    assert np.allclose(U.T @ U, np.eye(16), atol=1e-12)
    q = x.q.astype(np.float64).reshape(-1, x.d)
    frac = np.sum((q @ U) ** 2) / np.sum(q * q)  # energy of q inside span(U)
    assert frac > 0.5
    v = x.v_f32().astype(np.float64)
    assert abs(v.var() - 1.0) < 0.05


def test_cfg4_per_channel_log_uniform_scales():
    x = make_inputs("cfg4", B=1, Hkv=2, Hq=16, T=4096)
    for tens, key in ((x.k_f32(), "k_std"), (x.v_f32(), "v_std")):
        std = x.extra[key]
        assert std.shape == (x.Hkv, x.d) and np.all(std >= 0.1) and np.all(std <= 10.0)
        # log-uniform over two decades: log10 std uniform on [-1, 1]
        l10 = np.log10(std).ravel()
        assert abs(l10.mean()) < 0.15 and abs(l10.var() - 1.0 / 3.0) < 0.1
        emp = tens.astype(np.float64).std(axis=2)  # [B][Hkv][d]
        assert np.allclose(emp[0], std, rtol=0.06)


def test_cfg5_queries_in_a_per_head_subspace():
    x = make_inputs("cfg5", B=2, Hkv=2, Hq=8, T=64)
    A = x.extra["A"]
    G = x.Hq // x.Hkv
    assert A.shape == (x.Hkv, x.d, 24)
    for h in range(x.Hkv):
        assert np.allclose(A[h].T @ A[h], np.eye(24), atol=1e-12)
        qh = x.q[:, h * G:(h + 1) * G].reshape(-1, x.d).astype(np.float64)
        assert np.sum((qh @ A[h]) ** 2) / np.sum(qh * qh) > 0.85  # 24 of 128 dims, noise 0.01
        cal = x.extra["calib"][h]
        assert cal.shape == (CONFIGS["cfg5"]["calib"], x.d)
        s = _svals(cal)
        assert s[23] > 5 * s[24]


def test_sq_rank16_keys_values_and_separate_calibration():
    x = make_inputs("sq", B=1, Hkv=2, Hq=8, T=2048)
    for h in range(x.Hkv):
        for t, U, cal in ((x.k_f32()[0, h], x.extra["UK"][h], x.extra["calib_k"][h]),
                          (x.v_f32()[0, h], x.extra["UV"][h], x.extra["calib_v"][h])):
            s = _svals(t)
            assert s[15] > 5 * s[16]
            P = U @ U.T
            resid = np.asarray(t, dtype=np.float64) - np.asarray(t, dtype=np.float64) @ P
            assert np.sum(resid ** 2) / np.sum(np.asarray(t, dtype=np.float64) ** 2) < 0.15
            assert cal.shape == (CONFIGS["sq"]["calib"], x.d)
            assert _svals(cal)[15] > 5 * _svals(cal)[16]
    # keys and values use different subspaces
    cos = np.linalg.svd(x.extra["UK"][0].T @ x.extra["UV"][0], compute_uv=False)
    assert np.max(cos) < 0.9
