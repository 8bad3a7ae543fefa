"""Pins for the oracle's generator tables and rotation (no GPU)."""

import itertools

import numpy as np
from scipy import stats

from oracle import rotation, tables


def test_splitmix64_published_outputs():
    # SplitMix64 from state 0 (Steele, Lea & Flood 2014; the reference C implementation's
    # first three outputs): mix64(k * gamma) for k = 1, 2, 3.
    expected = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    got = [tables.mix64((k * tables.GAMMA) & tables.MASK64) for k in (1, 2, 3)]
    assert got == expected


def test_stream_is_splitmix_from_keyed_state():
    seed, stream = 12345, 3
    state = seed ^ tables.mix64(stream)
    h = tables.draws(seed, stream, 5)
    s = state
    for i in range(5):
        s = (s + tables.GAMMA) & tables.MASK64
        assert h[i] == tables.mix64(s)


def test_rotation_signs_balanced():
    D = tables.rotation_signs(7, tables.STREAM_D_K, 8192)
    assert set(np.unique(D)) == {-1.0, 1.0}
    assert stats.binomtest(int((D > 0).sum()), len(D)).pvalue > 1e-3
    assert not np.array_equal(D, tables.rotation_signs(7, tables.STREAM_D_V, 8192))


def test_sketch_entries_standard_normal():
    S = tables.sketch_matrix(0, tables.STREAM_S_K, 64, 512)
    assert S.dtype == np.float32 and S.shape == (64, 512)
    x = S.astype(np.float64).ravel()
    assert stats.kstest(x, "norm").pvalue > 1e-3
    assert abs(x.mean()) < 4 / np.sqrt(x.size) and abs(x.var() - 1) < 0.03


def test_hadamard_explicit_8():
    h2 = np.array([[1, 1], [1, -1]], dtype=np.float64)
    h8 = np.kron(np.kron(h2, h2), h2)  # Sylvester construction
    assert np.array_equal(rotation.sylvester_hadamard(8), h8)


def test_hadamard_recursion_and_orthogonality():
    for k in range(1, 11):
        d = 1 << k
        H = rotation.sylvester_hadamard(d)
        assert np.array_equal(H @ H.T, d * np.eye(d))
        if d >= 2:
            h = rotation.sylvester_hadamard(d // 2)
            assert np.array_equal(H, np.block([[h, h], [h, -h]]))


def test_rotation_orthogonal_and_norm_preserving():
    rng = np.random.default_rng(0)
    for d in (8, 128, 1024):
        D = tables.rotation_signs(1, tables.STREAM_D_K, d)
        R = rotation.rotation_matrix(D)
        assert np.allclose(R @ R.T, np.eye(d), atol=1e-13)
        # inverse is D H / sqrt(d)
        Rinv = np.diag(D) @ rotation.sylvester_hadamard(d) / np.sqrt(d)
        assert np.allclose(Rinv @ R, np.eye(d), atol=1e-13)
        x = rng.standard_t(1.5, size=d)
        assert abs(np.linalg.norm(R @ x) - np.linalg.norm(x)) < 1e-14 * np.linalg.norm(x) * 10


def test_rotated_coordinate_second_moment_exact_over_all_signs():
    # for any fixed unit x, averaging y_i^2 over all 2^d sign patterns gives exactly 1/d
    d = 8
    rng = np.random.default_rng(1)
    x = rng.standard_t(1.2, size=d)
    x /= np.linalg.norm(x)
    acc = np.zeros(d)
    for signs in itertools.product((-1.0, 1.0), repeat=d):
        acc += (rotation.rotation_matrix(np.array(signs)) @ x) ** 2
    assert np.allclose(acc / 2 ** d, 1.0 / d, atol=1e-15)
