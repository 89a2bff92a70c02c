"""Pins of the oracle's router: softmax, top-k order and gate weights (no GPU)."""
import math

import numpy as np
import pytest
import scipy.special

import oracle


def _logits(rng, E, d):
    w = rng.normal(0, 0.3, size=(E, d)).astype(np.float32)
    b = rng.normal(0, 0.1, size=E).astype(np.float32)
    x = rng.normal(0, 1, size=d).astype(np.float32)
    return w, b, x


@pytest.mark.parametrize("E,k", [(5, 2), (8, 3), (7, 7), (1, 1)])
def test_topk_matches_python_sort(E, k):
    rng = np.random.default_rng(E * 10 + k)
    for _ in range(20):
        w, b, x = _logits(rng, E, 16)
        logits, probs, sel, g = oracle.router(x, w, b, k)
        # brute force: Python sorted() over (-logit, index), logits from scalar loops
        lg = [sum(float(w[e, j]) * float(x[j]) for j in range(16)) + float(b[e]) for e in range(E)]
        order = [e for _, e in sorted((-lg[e], e) for e in range(E))][:k]
        assert list(sel) == order
        np.testing.assert_allclose(logits, lg, rtol=1e-12, atol=1e-12)


def test_softmax_matches_library():
    rng = np.random.default_rng(1)
    w, b, x = _logits(rng, 9, 12)
    logits, probs, sel, g = oracle.router(x, w, b, 4)
    np.testing.assert_allclose(probs, scipy.special.softmax(logits), rtol=1e-14)
    assert abs(probs.sum() - 1.0) < 1e-15
    np.testing.assert_allclose(g, probs[sel], rtol=0)


def test_two_experts_closed_form():
    w = np.array([[1.0, 0.0], [0.0, 1.0]], np.float32)
    x = np.array([0.7, -0.4], np.float32)
    _, probs, sel, g = oracle.router(x, w, None, 1)
    l0, l1 = float(x[0]), float(x[1])
    assert list(sel) == [0]
    assert math.isclose(g[0], 1.0 / (1.0 + math.exp(l1 - l0)), rel_tol=1e-14)


def test_k_equals_e_selects_all_and_renorm_is_softmax():
    rng = np.random.default_rng(2)
    w, b, x = _logits(rng, 6, 10)
    logits, probs, sel, g = oracle.router(x, w, b, 6, renorm=True)
    assert sorted(sel) == list(range(6))
    assert list(sel) == list(np.argsort(-logits, kind="stable"))
    np.testing.assert_allclose(g, probs[sel], rtol=1e-14)


def test_renorm_sums_to_one():
    rng = np.random.default_rng(4)
    w, b, x = _logits(rng, 12, 10)
    _, probs, sel, g = oracle.router(x, w, b, 3, renorm=True)
    assert abs(g.sum() - 1.0) < 1e-14
    np.testing.assert_allclose(g, probs[sel] / probs[sel].sum(), rtol=1e-14)


def test_ties_go_to_lower_index():
    w = np.zeros((5, 3), np.float32)
    w[1] = w[3] = [1.0, 0.0, 0.0]
    x = np.array([2.0, 1.0, 1.0], np.float32)
    _, _, sel, _ = oracle.router(x, w, None, 3)
    assert list(sel) == [1, 3, 0]


def test_margin():
    w = np.eye(4, dtype=np.float32)
    x = np.array([0.5, 0.25, 0.2, -1.0], np.float32)
    assert math.isclose(oracle.topk_margin(x, w, None, 2), 0.25 - 0.2, rel_tol=1e-6)
    assert oracle.topk_margin(x, w, None, 4) == math.inf
