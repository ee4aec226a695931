"""Pins for the oracle's router: top-k on logits (ties to the lower id) and softmax weights."""
import math

import numpy as np
import pytest

import oracle


def brute_topk(row, k):
    order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
    return order[:k]


@pytest.mark.parametrize("E,k", [(4, 1), (4, 2), (8, 2), (8, 8), (16, 5), (128, 8), (256, 8)])
def test_topk_matches_sorting(E, k):
    rng = np.random.default_rng(E * 100 + k)
    for trial in range(20):
        lg = rng.standard_normal((3, E)).astype(np.float32)
        if trial % 3 == 0:   # many exact ties
            lg = np.round(lg * 2) / 2
        ids, w = oracle.router(lg, k)
        for t in range(3):
            assert list(ids[t]) == brute_topk(lg[t], k)


def test_softmax_closed_form():
    # softmax of (0, ln 2, ln 3) over all three experts is (1/6, 2/6, 3/6)
    lg = np.array([[0.0, math.log(2.0), math.log(3.0)]], dtype=np.float32)
    ids, w = oracle.router(lg, 3, weight_mode=0)
    assert list(ids[0]) == [2, 1, 0]
    # the fp32 logits are not exactly ln 2, ln 3: compare at fp32 input precision
    np.testing.assert_allclose(w[0], [0.5, 1 / 3, 1 / 6], rtol=1e-7)
    # mode 1 renormalises over the chosen k: top-2 of the same row -> 3/5, 2/5
    ids, w = oracle.router(lg, 2, weight_mode=1)
    np.testing.assert_allclose(w[0], [0.6, 0.4], rtol=1e-7)


def test_weights_mode0_is_softmax_over_all_experts():
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((5, 16)).astype(np.float32)
    ids, w = oracle.router(lg, 16, 0)     # choosing all: the weights are the whole softmax
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    ids2, w2 = oracle.router(lg, 4, 0)
    assert np.all(w2.sum(axis=1) < 1.0)   # a strict part of the distribution
    np.testing.assert_array_equal(w2, w[:, :4])


def test_weights_mode1_sum_to_one():
    rng = np.random.default_rng(8)
    lg = rng.standard_normal((6, 32)).astype(np.float32)
    ids, w = oracle.router(lg, 8, 1)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)


def test_all_equal_logits():
    lg = np.zeros((2, 8), dtype=np.float32)
    ids, w = oracle.router(lg, 3, 0)
    assert ids.tolist() == [[0, 1, 2], [0, 1, 2]]
    np.testing.assert_array_equal(w, np.full((2, 3), 1 / 8))


def test_shift_invariance_of_weights():
    rng = np.random.default_rng(9)
    # multiples of 2^-10 below 4 in magnitude: adding 64 is exact in fp32
    lg = (np.round(rng.standard_normal((4, 16)) * 1024) / 1024).astype(np.float32)
    _, w1 = oracle.router(lg, 4, 0)
    shifted = lg + np.float32(64.0)
    assert np.array_equal(shifted - np.float32(64.0), lg)
    _, w2 = oracle.router(shifted, 4, 0)
    np.testing.assert_allclose(w1, w2, rtol=1e-12)


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
def test_non_finite_rejected(bad):
    lg = np.zeros((2, 8), dtype=np.float32)
    lg[1, 3] = bad
    with pytest.raises(ValueError):
        oracle.router(lg, 2)
