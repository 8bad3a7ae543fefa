"""The quality report's metric functions on hand-checkable inputs (no GPU)."""

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import quality  # noqa: E402


def test_vector_errors():
    x = np.array([[3.0, 4.0], [1.0, 0.0]])
    rel, dirr = quality._vec_errors(x, x)
    assert rel == 0.0 and abs(dirr) < 1e-15
    xh = np.array([[3.0, 4.0], [0.0, 1.0]])  # second vector rotated by 90 degrees
    rel, dirr = quality._vec_errors(x, xh)
    assert rel == pytest.approx(2.0 / 26.0)
    assert dirr == pytest.approx(0.5)  # mean of (1 - 1, 1 - 0)
    rel, dirr = quality._vec_errors(x, 2 * x)  # pure scale error
    assert rel == pytest.approx(1.0) and abs(dirr) < 1e-15


def test_attention_metrics_identity_and_shift_invariance():
    rng = np.random.default_rng(0)
    B, Hkv, G, T, d = 1, 2, 2, 50, 8
    K = rng.standard_normal((B, Hkv, T, d))
    q = rng.standard_normal((B, Hkv * G, d))
    kl, top5 = quality._attention_metrics(q, K, K, d, G)
    assert abs(kl) < 1e-12 and top5 == 1.0
    # doubling every key doubles the logits: a sharper distribution (KL > 0), the same top-5
    kl2, top52 = quality._attention_metrics(q, K, 2 * K, d, G)
    assert kl2 > 0 and top52 == 1.0


def test_reference_output_is_softmax_average():
    rng = np.random.default_rng(1)
    B, Hkv, G, T, d = 1, 1, 1, 7, 4
    K = rng.standard_normal((B, Hkv, T, d))
    V = rng.standard_normal((B, Hkv, T, d))
    q = rng.standard_normal((B, 1, d))
    o = quality._reference_output(q, K, V, d, G)
    s = K[0, 0] @ q[0, 0] / 2.0
    p = np.exp(s - s.max())
    p /= p.sum()
    assert np.allclose(o[0, 0], p @ V[0, 0])
