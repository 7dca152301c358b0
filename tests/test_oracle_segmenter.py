"""The oracle's row segmenter against numpy's stable argsort (a library
routine the segmenter must agree with) and against its stated readings."""

import numpy as np
import pytest

import oracle


def _numpy_segments(ids):
    ids = np.asarray(ids, np.int64)
    perm = np.argsort(ids, kind="stable").astype(np.int32)
    keys = ids[perm]
    if keys.size == 0:
        return perm, np.array([0], np.int32), np.array([], np.int32)
    starts = np.concatenate([[0], np.nonzero(np.diff(keys))[0] + 1])
    offs = np.concatenate([starts, [keys.size]]).astype(np.int32)
    return perm, offs, keys[starts].astype(np.int32)


@pytest.mark.parametrize("seed,M,S", [(0, 1, 1), (1, 17, 3), (2, 300, 40), (3, 4096, 2048), (4, 64, 32)])
def test_matches_numpy_stable_argsort(seed, M, S):
    rng = np.random.default_rng(seed)
    ids = rng.integers(-1, S, size=M).astype(np.int32)
    got = oracle.segment_rows(ids, S)
    want = _numpy_segments(ids)
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


def test_edge_cases():
    perm, offs, adp = oracle.segment_rows([], 4)
    assert perm.size == 0 and offs.tolist() == [0] and adp.size == 0
    perm, offs, adp = oracle.segment_rows([-1, -1, -1], 4)
    assert perm.tolist() == [0, 1, 2] and offs.tolist() == [0, 3] and adp.tolist() == [-1]
    perm, offs, adp = oracle.segment_rows([2, 2, 0, 2], 3)
    assert perm.tolist() == [2, 0, 1, 3] and offs.tolist() == [0, 1, 4] and adp.tolist() == [0, 2]
    for bad in ([0, 3], [-2], [5]):
        with pytest.raises(ValueError):
            oracle.segment_rows(bad, 3)


def test_rows_from_segments_roundtrip():
    rng = np.random.default_rng(9)
    ids = rng.integers(-1, 12, size=500).astype(np.int32)
    perm, offs, adp = oracle.segment_rows(ids, 12)
    assert np.array_equal(oracle.rows_from_segments(500, offs, adp, perm), ids)
    # identity permutation over pre-sorted rows
    sorted_ids = np.sort(ids, kind="stable")
    _, offs2, adp2 = oracle.segment_rows(sorted_ids, 12)
    assert np.array_equal(oracle.rows_from_segments(500, offs2, adp2), sorted_ids)
