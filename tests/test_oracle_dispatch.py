"""Pins for the oracle's dispatch-side permute (CPU).

Pinned against the inverse map (src_row, from a library stable sort of the
routing ids) and against the combine it inverts: gathering the permuted rows
back with top_k = 1 and weight 1 returns every token's own row."""
import numpy as np

import oracle
from norm_quant_gb300.synth import f32_to_bf16_bits

RNG = np.random.Generator(np.random.PCG64(21))


def _setup(T=50, k=4, E=9, H=40):
    ids = np.stack([RNG.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[RNG.random((T, k)) < 0.2] = -1
    st, counts, offsets, row_map, src_row = oracle.build_row_map(ids, E)
    x = f32_to_bf16_bits(RNG.standard_normal((T, H)).astype(np.float32))
    return ids, row_map, src_row, int(offsets[E]), x


def test_permute_matches_the_inverse_map():
    ids, row_map, src_row, nv, x = _setup()
    st, xg = oracle.dispatch_permute(x, row_map, nv)
    assert st == 0
    k = row_map.shape[1]
    # independent derivation: stable sort by expert gives, for each row, its slot
    flat = ids.reshape(-1)
    order = np.argsort(np.where(flat >= 0, flat, 1 << 30), kind="stable")[:nv]
    assert np.array_equal(xg, x[order // k])
    assert np.array_equal(src_row, order)


def test_combine_inverts_the_permute():
    ids, row_map, src_row, nv, x = _setup(T=31, k=3, E=5, H=64)
    st, xg = oracle.dispatch_permute(x, row_map, nv)
    for j in range(row_map.shape[1]):
        keep = row_map[:, j] >= 0
        o = oracle.combine(xg, row_map[keep][:, j:j + 1], np.ones((int(keep.sum()), 1), np.float32),
                           outputs=("combined",))
        assert np.array_equal(o["combined"], x[keep])


def test_unnamed_rows_untouched_and_bad_rows_reported():
    ids, row_map, src_row, nv, x = _setup(T=8, k=2, E=3, H=16)
    st, xg = oracle.dispatch_permute(x, row_map, nv + 3, fill=0x7777)
    assert st == 0 and np.all(xg[nv:] == 0x7777)
    bad = row_map.copy()
    bad[0, 0] = nv + 3
    st, _ = oracle.dispatch_permute(x, bad, nv + 3)
    assert st == 1
