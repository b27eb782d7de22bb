"""Pins of the oracle's merged order for the expert-parallel layer
(oracle.ep_regroup), against a brute force built from labelled rows: every
received row carries (source rank q, local expert e, position j in the
sender's order); the merged order is the rows sorted by (e, q, j)."""
import itertools

import numpy as np
import pytest

import oracle


def brute(counts):
    P, nl = counts.shape
    labels = [(q, e, j) for q in range(P) for e in range(nl) for j in range(counts[q, e])]
    merged = sorted(range(len(labels)), key=lambda i: (labels[i][1], labels[i][0], labels[i][2]))
    offsets = [0]
    for e in range(nl):
        offsets.append(offsets[-1] + int(counts[:, e].sum()))
    return np.array(offsets), np.array(merged, dtype=np.int64)


CASES = [
    np.array([[2, 0, 3], [1, 4, 0]]),
    np.array([[0, 0], [0, 0], [0, 0]]),
    np.array([[5]]),
    np.array([[0, 1, 0, 2], [3, 0, 0, 0], [1, 1, 1, 1]]),
]


@pytest.mark.parametrize("counts", CASES + [np.random.default_rng(s).integers(0, 6, (4, 5))
                                            for s in range(5)])
def test_regroup_is_the_sort_by_expert_then_rank(counts):
    offsets, perm, inv = oracle.ep_regroup(counts)
    b_off, b_perm = brute(counts)
    np.testing.assert_array_equal(offsets, b_off)
    np.testing.assert_array_equal(perm, b_perm)
    np.testing.assert_array_equal(inv[perm], np.arange(perm.size))


def test_regroup_single_rank_is_identity():
    for counts in itertools.product(range(3), repeat=3):
        offsets, perm, inv = oracle.ep_regroup(np.array([counts]))
        np.testing.assert_array_equal(perm, np.arange(sum(counts)))
        np.testing.assert_array_equal(inv, np.arange(sum(counts)))


def test_regroup_rejects_negative_counts():
    with pytest.raises(ValueError):
        oracle.ep_regroup(np.array([[1, -1]]))
