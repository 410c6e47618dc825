"""Pins for the oracle's dispatch (histogram, scan, stable packing), CPU only."""
import numpy as np
import pytest

from oracle import dispatch


def _check_invariants(idx, E):
    T, k = idx.shape
    R = T * k
    counts, offsets, pos, src = dispatch(idx, E)
    flat = idx.reshape(-1)
    assert counts.sum() == R
    assert offsets[0] == 0 and offsets[-1] == R
    assert np.array_equal(np.diff(offsets), counts)
    # pos is a permutation of 0..R-1
    assert np.array_equal(np.sort(pos), np.arange(R))
    # each entry lands inside its expert's segment
    for i in range(R):
        e = flat[i]
        assert offsets[e] <= pos[i] < offsets[e + 1]
    # stability: within one expert, positions grow with the flat index
    for e in range(E):
        p = pos[flat == e]
        assert np.all(np.diff(p) > 0)
    # src inverts pos; gathering rows by src and scattering back restores order
    assert np.array_equal(src[pos], np.arange(R) // k)
    rows = np.arange(T) * 10 + 3            # stand-in token rows
    packed = rows[src]
    assert np.array_equal(packed[pos].reshape(T, k), np.repeat(rows[:, None], k, 1))
    # brute force: a stable argsort of the expert ids is the inverse of pos
    order = np.argsort(flat, kind="stable")
    assert np.array_equal(pos[order], np.arange(R))
    return counts, offsets, pos, src


@pytest.mark.parametrize("seed", range(5))
def test_random_routing(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 40))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.integers(1, 60))
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    _check_invariants(idx, E)


def test_skew_and_empty_experts():
    idx = np.zeros((50, 1), dtype=np.int32)
    idx[10:12, 0] = 3
    counts, offsets, pos, src = _check_invariants(idx, 6)
    assert list(counts) == [48, 0, 0, 2, 0, 0]
    assert list(offsets) == [0, 48, 48, 48, 50, 50, 50]
    assert pos[10] == 48 and pos[11] == 49


def test_tiny_handworked():
    # tokens 0..2, top-2: (1,0), (0,2), (1,2)
    idx = np.array([[1, 0], [0, 2], [1, 2]])
    counts, offsets, pos, src = _check_invariants(idx, 3)
    assert list(counts) == [2, 2, 2]
    assert list(pos) == [2, 0, 1, 4, 3, 5]
    assert list(src) == [0, 1, 0, 2, 1, 2]


def test_empty_batch():
    idx = np.zeros((0, 2), dtype=np.int32)
    counts, offsets, pos, src = dispatch(idx, 4)
    assert counts.sum() == 0 and list(offsets) == [0] * 5 and pos.size == 0


def test_out_of_range_index_rejected():
    with pytest.raises(ValueError):
        dispatch(np.array([[0, 4]]), 4)
