"""Pins of the oracle router (CPU only): k = E is the full softmax (scipy),
all-equal logits pick experts 0..k-1 with weight 1/k, brute force over a
Python sort of (-logit, index) on tiny inputs, and non-finite handling."""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

from oracle import router


def test_k_equals_e_is_full_softmax():
    rng = np.random.default_rng(10)
    logits = rng.standard_normal((7, 12)).astype(np.float32)
    for renorm in (True, False):
        ids, w, flags = router.route_topk(logits, 12, renorm)
        assert not flags.any()
        p = softmax(logits.astype(np.float64), axis=1)
        for t in range(7):
            assert sorted(ids[t].tolist()) == list(range(12))
            np.testing.assert_allclose(w[t], p[t, ids[t]], rtol=1e-14, atol=0)
            # slots in descending probability
            assert np.all(np.diff(p[t, ids[t]]) <= 0)


def test_all_equal_logits_pick_lowest_indices():
    logits = np.full((3, 16), 0.375, dtype=np.float32)
    ids, w, _ = router.route_topk(logits, 5, True)
    np.testing.assert_array_equal(ids, np.tile(np.arange(5), (3, 1)))
    np.testing.assert_allclose(w, 0.2, rtol=1e-15)
    ids, w, _ = router.route_topk(logits, 5, False)
    np.testing.assert_allclose(w, 1 / 16, rtol=1e-15)


def test_brute_force_tiny():
    rng = np.random.default_rng(11)
    for trial in range(200):
        E = int(rng.integers(1, 9))
        k = int(rng.integers(1, E + 1))
        # few distinct values -> many ties
        logits = rng.integers(-2, 3, size=(1, E)).astype(np.float32) * np.float32(0.5)
        ids, w, _ = router.route_topk(logits, k, True)
        order = sorted(range(E), key=lambda e: (-float(logits[0, e]), e))
        assert ids[0].tolist() == order[:k]
        ex = np.exp(logits[0].astype(np.float64))
        sel = ex[order[:k]]
        np.testing.assert_allclose(w[0], sel / sel.sum(), rtol=1e-14)


def test_top1_is_argmax():
    rng = np.random.default_rng(12)
    logits = rng.standard_normal((50, 64)).astype(np.float32)
    ids, w, _ = router.route_topk(logits, 1, True)
    np.testing.assert_array_equal(ids[:, 0], np.argmax(logits, axis=1))
    np.testing.assert_array_equal(w, 1.0)


def test_nonfinite_rank_last_with_zero_weight():
    logits = np.array([[0.5, np.nan, -np.inf, 2.0, np.inf, -1.0]], dtype=np.float32)
    ids, w, flags = router.route_topk(logits, 6, False)
    assert flags[0]
    assert ids[0].tolist() == [3, 0, 5, 1, 2, 4]
    fin = np.array([2.0, 0.5, -1.0])
    p = np.exp(fin) / np.exp(fin).sum()
    np.testing.assert_allclose(w[0, :3], p, rtol=1e-14)
    np.testing.assert_array_equal(w[0, 3:], 0.0)
    ids, w, _ = router.route_topk(np.full((1, 4), np.nan, np.float32), 2, True)
    assert ids[0].tolist() == [0, 1]
    np.testing.assert_array_equal(w, 0.0)


def test_bad_k():
    with pytest.raises(ValueError):
        router.route_topk(np.zeros((1, 4), np.float32), 5)
