"""Pins of the HeadQ calibration basis (oracle/headq.py ``calibration_basis``): the top-r principal
directions of the centred sample covariance of a KV head's calibration queries ([HEADQ] "Visão
Geral do Algoritmo" 1).

Eigenvectors are unique only up to sign (and within degenerate eigenspaces), so every check
compares what is unique: the projector U U^T, the captured variance, orthonormality.  None of
them calls an eigen-solver: maximality is checked against random frames (Ky Fan), the subspace
against a planted one, and the leading direction at d = 2 by brute force over angles."""

import numpy as np
import pytest

from oracle import headq


def _planted(n, d, r, rng, spread=(9.0, 1.5), noise=0.05, mean=None):
    A, _ = np.linalg.qr(rng.standard_normal((d, r)))
    sig = np.linspace(spread[0], spread[1], r)  # distinct variances: no degenerate subspace
    X = (rng.standard_normal((n, r)) * sig) @ A.T + noise * rng.standard_normal((n, d))
    if mean is not None:
        X = X + mean
    return X, A


def _cov(X):
    Xc = X - X.mean(axis=0, keepdims=True)
    return Xc.T @ Xc / (X.shape[0] - 1)


def test_orthonormal_columns():
    rng = np.random.default_rng(1)
    X, _ = _planted(3000, 64, 12, rng)
    U = headq.calibration_basis(X, 12)
    assert U.shape == (64, 12)
    assert np.allclose(U.T @ U, np.eye(12), atol=1e-12)


@pytest.mark.parametrize("r", [1, 4, 16])
def test_recovers_a_planted_subspace(r):
    rng = np.random.default_rng(2 + r)
    X, A = _planted(6000, 128, r, rng)
    U = headq.calibration_basis(X, r)
    # principal-angle cosines between span(U) and span(A): all near 1
    cos = np.linalg.svd(A.T @ U, compute_uv=False)
    assert np.min(cos) > 0.999


def test_captures_more_variance_than_any_other_frame():
    # Ky Fan: tr(U^T C U) is the largest over orthonormal r-frames; random frames and perturbed
    # copies of U must not beat it
    rng = np.random.default_rng(3)
    d, r = 48, 6
    X, _ = _planted(4000, d, r, rng, spread=(5.0, 0.8), noise=0.3)
    C = _cov(X)
    U = headq.calibration_basis(X, r)
    best = np.trace(U.T @ C @ U)
    for _ in range(200):
        V, _ = np.linalg.qr(rng.standard_normal((d, r)))
        assert np.trace(V.T @ C @ V) <= best + 1e-12
    for eps in (1e-3, 1e-2, 1e-1):
        V, _ = np.linalg.qr(U + eps * rng.standard_normal((d, r)))
        assert np.trace(V.T @ C @ V) <= best + 1e-12


def test_mean_is_removed_and_scale_does_not_matter():
    # a large common offset (an uncentred second moment would put the mean direction first)
    rng = np.random.default_rng(4)
    d, r = 32, 3
    X, A = _planted(5000, d, r, rng)
    g = rng.standard_normal(d)
    g -= A @ (A.T @ g)  # an offset outside the planted subspace
    mu = 40.0 * g / np.linalg.norm(g)
    P = lambda U: U @ U.T
    U0 = headq.calibration_basis(X, r)
    assert np.allclose(P(headq.calibration_basis(X + mu, r)), P(U0), atol=1e-9)
    assert np.allclose(P(headq.calibration_basis(7.5 * X, r)), P(U0), atol=1e-9)
    # the offset's direction, the leading one of the uncentred second moment, is not in the basis
    m = mu / np.linalg.norm(mu)
    assert np.linalg.norm(headq.calibration_basis(X + mu, r).T @ m) < 0.05


def test_leading_direction_by_brute_force_in_two_dimensions():
    rng = np.random.default_rng(5)
    th = 0.7
    R = np.array([[np.cos(th), -np.sin(th)], [np.sin(th), np.cos(th)]])
    X = (rng.standard_normal((20000, 2)) * np.array([3.0, 1.0])) @ R.T + np.array([5.0, -2.0])
    C = _cov(X)
    grid = np.linspace(0.0, np.pi, 200001)
    dirs = np.stack([np.cos(grid), np.sin(grid)], axis=1)
    rq = np.einsum("ni,ij,nj->n", dirs, C, dirs)  # Rayleigh quotient over all directions
    u = dirs[np.argmax(rq)]
    U = headq.calibration_basis(X, 1)
    assert abs(float(U[:, 0] @ u)) > 1 - 1e-9
