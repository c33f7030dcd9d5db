"""Pins for the oracle's top-K cache producer: brute force on tiny inputs (a
plain Python sort of every (logit, id) pair), ties broken by the smaller id,
and agreement with numpy's argpartition on random data."""
import math

import numpy as np
import pytest

import oracle.kl_oracle as ok


def _brute(z, K):
    out = []
    for row in z:
        pairs = sorted(((-float(v), i) for i, v in enumerate(row)))
        out.append([i for _, i in pairs[:K]])
    return np.array(out)


@pytest.mark.parametrize("K", [1, 3, 7])
def test_matches_brute_force(K):
    rng = np.random.default_rng(K)
    H = rng.standard_normal((5, 4))
    W = rng.standard_normal((9, 4))
    ids, vals = ok.topk_logits(H, W, K)
    z = H @ W.T
    np.testing.assert_array_equal(ids, _brute(z, K))
    np.testing.assert_array_equal(vals, np.take_along_axis(z, ids, axis=1))
    assert (np.diff(vals, axis=1) <= 0).all()


def test_ties_take_smaller_id():
    H = np.array([[1.0, 0.0]])
    W = np.array([[1.0, 0.0], [2.0, 0.0], [1.0, 5.0], [2.0, -1.0], [1.0, 0.0]])
    ids, vals = ok.topk_logits(H, W, 4)
    assert ids.tolist() == [[1, 3, 0, 2]]  # values 2, 2, 1, 1 (ids 0, 2, 4 tie at 1)
    assert vals.tolist() == [[2.0, 2.0, 1.0, 1.0]]


def test_against_argpartition():
    rng = np.random.default_rng(0)
    H = rng.standard_normal((30, 16))
    W = rng.standard_normal((500, 16)) / 4
    K = 25
    ids, vals = ok.topk_logits(H, W, K)
    z = H @ W.T
    part = np.argpartition(-z, K - 1, axis=1)[:, :K]
    for t in range(30):
        assert set(ids[t]) == set(part[t])
        assert math.isclose(vals[t, -1], np.sort(z[t])[-K])


def test_k_equals_v_is_full_sort():
    rng = np.random.default_rng(1)
    H = rng.standard_normal((3, 5))
    W = rng.standard_normal((6, 5))
    ids, vals = ok.topk_logits(H, W, 6)
    for t in range(3):
        assert sorted(ids[t]) == list(range(6))
    assert (np.diff(vals, axis=1) <= 0).all()
