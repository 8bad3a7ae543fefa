"""Statistical pins of the oracle: Beta marginal, QJL estimator, variance inflation, Jensen (no GPU)."""

import os

import numpy as np
import pytest
from scipy import stats

from oracle import codebook, codec, rotation, tables

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _claims():
    out = {}
    for line in open(os.path.join(GOLDEN, "qjl_variance_claims.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            out[k] = float(v)
    return out


@pytest.mark.parametrize("d,n", [(8, 100000), (128, 100000), (1024, 20000)])
def test_rotated_unit_vector_coordinate_is_beta(d, n):
    # [TQ-KV] "Marco Teórico": (u_1 + 1)/2 ~ Beta((d-1)/2, (d-1)/2) for u uniform on the sphere
    rng = np.random.default_rng(d)
    R = rotation.rotation_matrix(tables.rotation_signs(3, tables.STREAM_D_K, d))
    samples = np.empty(n)
    chunk = 5000
    for s in range(0, n, chunk):
        g = rng.standard_normal((min(chunk, n - s), d))
        u = g / np.linalg.norm(g, axis=1, keepdims=True)
        y = u @ R.T
        samples[s:s + len(g)] = y[np.arange(len(g)), rng.integers(0, d, len(g))]
    assert stats.kstest(samples, lambda x: codebook.cdf(x, d)).pvalue > 1e-3


def _qjl_trials(q, r, m, trials, rng):
    d = len(q)
    est = np.empty(trials)
    rho = np.linalg.norm(r)
    for i in range(trials):
        S = rng.standard_normal((m, d))
        est[i] = codec.qjl_inner_product(q, S, rho, (S @ r) >= 0)
    return est


@pytest.mark.parametrize("d", [8, 128])
def test_qjl_unbiased_with_stated_variance(d):
    # [TQ-KV] "Contribuciones Clave" 1: unbiased residual estimator, variance (pi/2)||r||^2/d
    rng = np.random.default_rng(11 + d)
    m = d
    q = rng.standard_normal(d)
    q /= np.linalg.norm(q)
    r = 0.1 * rng.standard_normal(d)
    trials = 10000
    est = _qjl_trials(q, r, m, trials, rng)
    truth = q @ r
    se = est.std() / np.sqrt(trials)
    assert abs(est.mean() - truth) < 4 * se
    exact_var = (np.pi / 2 * (q @ q) * (r @ r) - truth ** 2) / m
    assert abs(est.var() / exact_var - 1) < 0.05
    # the page's figure for unit q: (pi/2) * ||r||^2 / d, up to the <q, r>^2 / m term
    page = _claims()["qjl_estimator_variance_factor"] * (r @ r) / d
    assert abs(est.var() - page) <= truth ** 2 / m + 0.05 * page


def test_qjl_inflation_at_least_half_pi():
    # the sketch estimate of <q, r> has at least pi/2 times the variance of <q, r> itself
    # over random unit q ([TQ-KV] "Contribuciones Clave" 1)
    rng = np.random.default_rng(5)
    d = m = 64
    r = rng.standard_normal(d)
    qs = rng.standard_normal((4000, d))
    qs /= np.linalg.norm(qs, axis=1, keepdims=True)
    err = np.empty(len(qs))
    for i, q in enumerate(qs):
        S = rng.standard_normal((m, d))
        err[i] = codec.qjl_inner_product(q, S, np.linalg.norm(r), (S @ r) >= 0) - q @ r
    base = np.mean((qs @ r) ** 2)
    ratio = np.mean(err ** 2) / base
    assert ratio > _claims()["qjl_vs_scalar_residual_min"] * 0.9


def test_nbit_scalar_vs_nminus1_plus_qjl_ratio_near_two_pi():
    # [TQ-KV] "Contribuciones Clave" 1: (n-1)-bit + 1-bit QJL inflates the inner-product
    # error variance ~2*pi-fold over an n-bit scalar code (a high-rate figure; loose check)
    rng = np.random.default_rng(9)
    d, n = 128, 4
    R = rotation.rotation_matrix(tables.rotation_signs(1, tables.STREAM_D_K, d))
    cn, tn = codebook.fp32_tables(d, n)
    cm, tm = codebook.fp32_tables(d, n - 1)
    e_scalar, e_qjl = [], []
    for _ in range(3000):
        x = rng.standard_normal(d)
        q = rng.standard_normal(d)
        S = rng.standard_normal((d, d)).astype(np.float32)
        f_n = codec.encode(x[None], codec.SideCodec(n, True, False), cn, tn, R)
        f_q = codec.encode(x[None], codec.SideCodec(n - 1, True, True), cm, tm, R, S)
        xn = codec.reconstruct(codec.SideCodec(n, True, False), f_n["codes"], f_n["norm"], cn, R)
        xq = codec.reconstruct(codec.SideCodec(n - 1, True, True), f_q["codes"], f_q["norm"], cm, R,
                               f_q["rho"], f_q["signs"], S)
        e_scalar.append(q @ (xn[0] - x))
        e_qjl.append(q @ (xq[0] - x))
    ratio = np.var(e_qjl) / np.var(e_scalar)
    target = _claims()["nbit_vs_nminus1_plus_qjl"]
    assert 0.75 * target < ratio < 1.25 * target, ratio


def test_jensen_amplification():
    # [ABL] "Contribuições Principais" 2: E[exp(s + eps)] = exp(s) exp(sigma^2 / 2), eps ~ N(0, sigma^2)
    rng = np.random.default_rng(2)
    s, sigma = 0.7, 0.5
    eps = rng.normal(0, sigma, 2_000_000)
    mc = np.mean(np.exp(s + eps))
    assert abs(mc / (np.exp(s) * np.exp(sigma ** 2 / 2)) - 1) < 3e-3
