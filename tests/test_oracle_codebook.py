"""Pins for the oracle's Beta Lloyd-Max codebook (no GPU).

Each test checks the oracle against something other than itself: closed forms,
independent numerical quadrature, a published table, brute force.
"""

import os

import numpy as np
import pytest
from scipy import integrate, special

from oracle import codebook

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _quad(f, lo, hi, d):
    # split at the density's bulk so quad resolves the narrow peak for large d
    w = min(1.0, 12.0 / np.sqrt(d))
    pts = [p for p in (-w, 0.0, w) if lo < p < hi]
    return integrate.quad(f, lo, hi, points=pts or None, limit=400, epsabs=1e-15, epsrel=1e-13)[0]


@pytest.mark.parametrize("d", [8, 128, 1024])
def test_density_normalized_and_second_moment(d):
    # a unit vector's coordinates have E[u_1^2] = 1/d; the density must integrate to 1
    f = lambda x: codebook.density(x, d)
    assert abs(_quad(f, -1, 1, d) - 1.0) < 1e-11
    assert abs(_quad(lambda x: x * x * codebook.density(x, d), -1, 1, d) - 1.0 / d) < 1e-12


@pytest.mark.parametrize("d", [8, 128, 1024])
def test_one_bit_is_mean_absolute_coordinate(d):
    # b = 1: the two centroids are +-E|u_1| = Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2))
    c, t = codebook.lloyd_max(d, 1)
    expected = np.exp(special.gammaln(d / 2) - special.gammaln((d + 1) / 2)) / np.sqrt(np.pi)
    assert np.allclose(c, [-expected, expected], atol=1e-14, rtol=0)
    assert t[0] == 0.0


@pytest.mark.parametrize("d", [8, 128, 1024])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_lloyd_conditions_by_independent_quadrature(d, bits):
    # centroid = conditional mean of its cell, threshold = midpoint, computed by adaptive quadrature
    c, t = codebook.lloyd_max(d, bits)
    assert np.all(np.diff(c) > 0)
    assert np.allclose(c, -c[::-1], atol=0, rtol=0)
    assert np.allclose(t, 0.5 * (c[:-1] + c[1:]), atol=1e-16)
    edges = np.concatenate([[-1.0], t, [1.0]])
    for k in range(len(c)):
        m0 = _quad(lambda x: codebook.density(x, d), edges[k], edges[k + 1], d)
        m1 = _quad(lambda x: x * codebook.density(x, d), edges[k], edges[k + 1], d)
        assert abs(m1 / m0 - c[k]) < 1e-11 / np.sqrt(d) * 10, (k, m1 / m0, c[k])


def test_gaussian_limit_matches_max_1960():
    # sqrt(d) * c tends to the Gaussian Lloyd-Max levels (published table)
    rows = [l.split() for l in open(os.path.join(GOLDEN, "max1960_gaussian_lloyd_max.txt"))
            if l.strip() and not l.startswith("#")]
    d = 1 << 18
    for row in rows:
        L, mse = int(row[0]), float(row[1])
        pos = np.array([float(v) for v in row[2:]])
        bits = L.bit_length() - 1
        c, t = codebook.lloyd_max(d, bits)
        assert np.allclose(np.sqrt(d) * c[L // 2:], pos, atol=1.5e-3), (L, np.sqrt(d) * c[L // 2:])
        assert abs(codebook.mse(c, t, d) * d - mse) < 2e-4 * max(1.0, mse * 10)


@pytest.mark.parametrize("bits", [1, 2])
def test_brute_force_d8(bits):
    # grid search over odd-symmetric codebooks with nearest-neighbour cells; MSE by quadrature
    d = 8
    c_lm, t_lm = codebook.lloyd_max(d, bits)
    xs = np.linspace(-1, 1, 400001)
    w = codebook.density(xs, d)
    w /= w.sum()

    def mse_of(levels):
        levels = np.sort(np.concatenate([-levels, levels]))
        idx = np.abs(xs[:, None] - levels[None, :]).argmin(axis=1)
        return np.sum(w * (xs - levels[idx]) ** 2)

    if bits == 1:
        grid = np.linspace(0.2, 0.4, 401)
        best = grid[np.argmin([mse_of(np.array([g])) for g in grid])]
        assert abs(best - c_lm[1]) < 1e-3
    else:
        g1 = np.linspace(0.1, 0.25, 61)
        g2 = np.linspace(0.4, 0.65, 61)
        vals = np.array([[mse_of(np.array([a, b])) for b in g2] for a in g1])
        i, j = np.unravel_index(np.argmin(vals), vals.shape)
        assert abs(g1[i] - c_lm[2]) < 5e-3 and abs(g2[j] - c_lm[3]) < 5e-3
        assert vals[i, j] >= codebook.mse(c_lm, t_lm, d) - 1e-6


@pytest.mark.parametrize("d", [8, 128, 1024])
def test_mse_decreases_with_bits(d):
    errs = [codebook.mse(*codebook.lloyd_max(d, b), d) for b in (1, 2, 3, 4)]
    assert all(errs[i + 1] < errs[i] for i in range(3))
    assert errs[0] < 1.0 / d  # any codebook beats predicting 0


def test_cdf_matches_quadrature():
    d = 128
    for x in (-0.3, -0.05, 0.0, 0.02, 0.2):
        assert abs(codebook.cdf(x, d) - _quad(lambda u: codebook.density(u, d), -1, x, d)) < 1e-12
        assert abs(codebook.survival(x, d) - (1 - codebook.cdf(x, d))) < 1e-14
