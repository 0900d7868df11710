"""Pins for the oracle's routing build (CPU only).

The oracle counts and scatters in one pass over (t, j); the pin is a
different algorithm: a library stable sort of the valid entries by expert id,
whose output order is by definition the expert-grouped, stable row order.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.Generator(np.random.PCG64(11))


def _by_stable_sort(ids: np.ndarray, E: int):
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    order = np.argsort(np.where(valid, flat, E), kind="stable")[: int(valid.sum())]
    row_map = np.full(flat.shape, -1, np.int64)
    row_map[order] = np.arange(order.size)
    counts = np.bincount(flat[valid], minlength=E)
    return counts, row_map.reshape(ids.shape), order


def _random_ids(T, k, E, pad_rows=0.0, dup=False, bad=False):
    if dup:
        ids = RNG.integers(0, E, (T, k))
    else:
        ids = np.stack([RNG.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), int)
    if pad_rows and T:
        ids[RNG.random(T) < pad_rows] = -1
    if T:
        ids[RNG.random((T, k)) < 0.05] = -1
    if bad and T:
        ids[0, 0] = E
        ids[-1, -1] = -7
    return ids.astype(np.int32)


@pytest.mark.parametrize("T,k,E,kw", [
    (1, 1, 1, {}), (16, 2, 8, {}), (64, 8, 16, {}), (50, 4, 4, {"dup": True}),
    (33, 3, 5, {"pad_rows": 0.3}), (40, 8, 256, {"pad_rows": 1.0}), (0, 4, 8, {}),
    (200, 6, 7, {"dup": True, "pad_rows": 0.1}),
])
def test_routing_matches_stable_sort(T, k, E, kw):
    ids = _random_ids(T, k, E, **kw)
    st, counts, offsets, row_map, src_row = oracle.build_row_map(ids, E)
    assert st == 0
    c_want, rm_want, order = _by_stable_sort(ids, E)
    assert np.array_equal(counts, c_want)
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), c_want)
    assert np.array_equal(row_map, rm_want)
    assert np.array_equal(src_row, order)


def test_routing_invariants():
    T, k, E = 300, 8, 32
    ids = _random_ids(T, k, E, dup=True, pad_rows=0.1)
    st, counts, offsets, row_map, src_row = oracle.build_row_map(ids, E)
    n_valid = int((ids >= 0).sum())
    assert counts.sum() == n_valid == offsets[E]
    rows = row_map[row_map >= 0]
    assert np.array_equal(np.sort(rows), np.arange(n_valid))       # bijection
    for e in range(E):
        r = row_map[ids == e]                                       # (t, j) order
        assert np.all(np.diff(r) == 1) and (r.size == 0 or r[0] == offsets[e])
    assert np.all(row_map[ids < 0] == -1)


def test_routing_invalid_ids_are_flagged_and_padded():
    ids = _random_ids(20, 4, 6, bad=True)
    st, counts, offsets, row_map, _ = oracle.build_row_map(ids, 6)
    assert st == 4
    assert row_map[0, 0] == -1 and row_map[-1, -1] == -1
    assert counts.sum() == int(((ids >= 0) & (ids < 6)).sum())


@pytest.mark.parametrize("bad", [6, 7, 1000, -2, -1000])
def test_each_kind_of_invalid_id_is_flagged_on_its_own(bad):
    """An id at or above E, or below -1, is reported even when it is the
    only invalid one; -1 alone is padding and is not."""
    ids = np.array([[0, 5], [bad, 1], [-1, 2]], np.int32)
    st, counts, _, row_map, _ = oracle.build_row_map(ids, 6)
    assert st == 4 and row_map[1, 0] == -1 and counts.sum() == 4
    st, _, _, _, _ = oracle.build_row_map(np.where(ids == bad, -1, ids).astype(np.int32), 6)
    assert st == 0
