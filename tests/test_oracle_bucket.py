"""Pins of the oracle bucketing (CPU only), by closed form: offsets are the
exclusive prefix sum of np.bincount over the kept ids, every kept pair appears
exactly once, and the pair list equals np.lexsort by (expert, pair number)."""
import numpy as np

from oracle import bucket as B


def closed_form(ids, E, keep):
    flat = ids.reshape(-1)
    kept = np.nonzero(keep)[0]
    counts = np.bincount(flat[kept], minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    pairs = kept[np.lexsort((kept, flat[kept]))]
    return offsets, pairs, np.nonzero(counts)[0]


def random_ids(rng, T, E, k):
    if T == 0:
        return np.zeros((0, k), np.int32)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


def test_closed_form_random():
    rng = np.random.default_rng(20)
    for _ in range(50):
        E = int(rng.integers(1, 40))
        k = int(rng.integers(1, E + 1))
        T = int(rng.integers(0, 30))
        ids = random_ids(rng, T, E, k).reshape(T, k)
        offsets, pairs, pos, active, flags = B.bucket(ids, E)
        off2, pairs2, act2 = closed_form(ids, E, np.ones(T * k, bool))
        np.testing.assert_array_equal(offsets, off2)
        np.testing.assert_array_equal(pairs, pairs2)
        np.testing.assert_array_equal(active, act2)
        assert flags == 0
        # pos inverts pairs; every pair exactly once
        np.testing.assert_array_equal(pos[pairs], np.arange(len(pairs)))
        assert sorted(pairs.tolist()) == list(range(T * k))


def test_skip_sentinel_and_bad_ids():
    ids = np.array([[3, -1], [-1, -1], [7, 0], [5, 3]], dtype=np.int32)
    offsets, pairs, pos, active, flags = B.bucket(ids, 6)
    assert flags & B.FLAG_BAD_ID            # id 7 >= E
    assert not flags & B.FLAG_DUPLICATE_ID
    # kept: p0 (3), p5 (0), p6 (5), p7 (3)
    np.testing.assert_array_equal(offsets, [0, 1, 1, 1, 3, 3, 4])
    np.testing.assert_array_equal(pairs, [5, 0, 7, 6])
    np.testing.assert_array_equal(pos, [1, -1, -1, -1, -1, 0, 3, 2])
    np.testing.assert_array_equal(active, [0, 3, 5])


def test_duplicate_flagged_but_bucketed():
    ids = np.array([[2, 2], [1, 0]], dtype=np.int32)
    offsets, pairs, pos, active, flags = B.bucket(ids, 4)
    assert flags & B.FLAG_DUPLICATE_ID
    np.testing.assert_array_equal(pairs, [3, 2, 0, 1])


def test_range_and_format_filters():
    rng = np.random.default_rng(21)
    E, k, T = 16, 4, 12
    ids = random_ids(rng, T, E, k)
    fmts = rng.integers(1, 5, E)
    for lo, hi, mask in [(0, 16, 0xFFFFFFFF), (4, 9, 0xFFFFFFFF), (0, 16, 1 << 2), (3, 12, (1 << 1) | (1 << 4))]:
        offsets, pairs, pos, active, _ = B.bucket(ids, E, lo, hi, mask, fmts)
        flat = ids.reshape(-1)
        keep = (flat >= lo) & (flat < hi) & (((mask >> fmts[flat]) & 1) == 1)
        off2, pairs2, act2 = closed_form(ids, E, keep)
        np.testing.assert_array_equal(offsets, off2)
        np.testing.assert_array_equal(pairs, pairs2)
        np.testing.assert_array_equal(active, act2)
        assert (pos >= 0).sum() == keep.sum()


def test_empty():
    offsets, pairs, pos, active, flags = B.bucket(np.zeros((0, 3), np.int32), 5)
    np.testing.assert_array_equal(offsets, np.zeros(6))
    assert len(pairs) == 0 and len(active) == 0 and flags == 0
