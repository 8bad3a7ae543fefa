"""The hand-built edge-case inputs (tests/edge_inputs.py) have the properties the GPU edge tests
rely on: exact unit norm with a coordinate exactly on each fp32 threshold (so the oracle's
decision there is the lower cell), and extreme-range vectors that really leave fp32's range."""

import numpy as np
import pytest

from oracle import codebook, codec
from tests.edge_inputs import exact_square_sum, extreme_vectors, tie_vectors
from workloads import bf16_to_f32


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_tie_vectors_sit_exactly_on_thresholds(bits):
    d = 128
    C, T = codebook.fp32_tables(d, bits)
    targets = list(T) + [0.0]
    positions = [0, 5, 64, 127]
    X = tie_vectors(targets, d, positions)
    assert X.dtype == np.float32
    for x in X:
        assert exact_square_sum(x) == 1
    o = codec.encode(X.astype(np.float64), codec.SideCodec(bits, False, False), C, T, np.eye(d))
    assert np.all(o["norm"] == np.float32(1.0))
    for i, t in enumerate(targets):
        for jp, pos in enumerate(positions):
            row = 4 * i + jp
            assert o["y"][row, pos].astype(np.float32) == np.float32(t)
            assert o["code_margin"][row, pos] < 1e-15  # float64 rounding of the norm only
            assert o["codes"][row, pos] == int(np.sum(T < np.float32(t)))  # the lower cell


def test_extreme_vectors_leave_the_fp32_range():
    rng = np.random.default_rng(0)
    X = bf16_to_f32(extreme_vectors(rng, 10, 128)).astype(np.float64)
    assert np.all(np.isfinite(X))
    sq32 = [np.sum(x.astype(np.float32) ** 2, dtype=np.float32) for x in X]
    with np.errstate(over="ignore"):
        assert not np.isfinite(sq32[0]) and not np.isfinite(sq32[1])  # huge coordinates overflow
    assert sq32[2] == 0.0                                  # every square underflows
    assert 0 < np.sum(X[3] ** 2) < np.finfo(np.float32).tiny * 128  # squares in the subnormal range
    nu = np.sqrt(np.sum(X ** 2, axis=1))
    assert np.all(nu > 0) and np.all(nu < np.finfo(np.float32).max)
