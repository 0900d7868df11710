"""The workspace-free routing build, for callers that cannot allocate device
memory (framework plug-ins that own no memory of their own, loops that may
not call cudaMalloc).  Called through the C ABI, it must give exactly what
the oracle and the regular entry point give, call after call, although every
call reuses the library's one fixed scratch array: a call after one that met
an invalid id must report a clean flag, and a call after a larger one on
another routing path must not see the histograms that call left behind.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""
import ctypes as C

import numpy as np
import pytest
import torch

import norm_quant_gb300 as nqg
import oracle
from norm_quant_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ids(rng, T, k, E, bad=False):
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, k)) < 0.1] = -1
    if bad:
        ids[T // 2, 0] = E + 3
    return ids


def _outputs(T, k, E):
    return (torch.full((E,), -9, dtype=torch.int32, device=DEV),
            torch.full((E + 1,), -9, dtype=torch.int32, device=DEV),
            torch.full((T, k), -9, dtype=torch.int32, device=DEV),
            torch.full((max(T * k, 1),), -9, dtype=torch.int32, device=DEV))


def _regular(ids, E):
    T, k = ids.shape
    counts, offsets, row_map, src_row = _outputs(T, k, E)
    ws = torch.zeros(nqg.moe_build_row_map_workspace_size(T, k, E), dtype=torch.uint8, device=DEV)
    nqg.moe_build_row_map(ids, E, counts, offsets, row_map, src_row, ws)
    return counts, offsets, row_map, src_row, nqg.moe_build_row_map_check(ws)


def _noalloc(ids, E):
    """The workspace-free entry point, called through ctypes with raw device
    pointers."""
    T, k = ids.shape
    counts, offsets, row_map, src_row = _outputs(T, k, E)
    flag = torch.full((1,), -9, dtype=torch.int32, device=DEV)
    st = nqg.lib().moe_build_row_map_noalloc(
        C.c_void_p(ids.data_ptr()), T, k, E, C.c_void_p(counts.data_ptr()), C.c_void_p(offsets.data_ptr()),
        C.c_void_p(row_map.data_ptr()), C.c_void_p(src_row.data_ptr()), C.c_void_p(flag.data_ptr()),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == nqg.MOE_OK, nqg.moe_status_string(st)
    torch.cuda.synchronize()
    return counts, offsets, row_map, src_row, int(flag.item())


def _check_one_call(ids_np, E, what):
    """One workspace-free build against the oracle (bit for bit) and the
    regular entry point on the same ids."""
    ids = torch.from_numpy(ids_np).to(DEV)
    c1, o1, r1, s1, flag = _noalloc(ids, E)
    ost, oc, oo, orm, osr = oracle.build_row_map(ids_np, E)
    assert np.array_equal(c1.cpu().numpy(), oc), what
    assert np.array_equal(o1.cpu().numpy(), oo), what
    assert np.array_equal(r1.cpu().numpy(), orm), what
    n_valid = int(oo[E])
    assert np.array_equal(s1.cpu().numpy()[:n_valid], osr), what
    assert (flag != 0) == (ost != 0), f"{what}: flag {flag}, oracle status {ost}"
    c0, o0, r0, s0, st0 = _regular(ids, E)
    assert torch.equal(c0, c1) and torch.equal(o0, o1) and torch.equal(r0, r1), what
    assert torch.equal(s0[:n_valid], s1[:n_valid]), what
    assert (st0 == nqg.MOE_ERR_INVALID_EXPERT) == (flag != 0), what
    return flag


@pytest.mark.parametrize("order", [("clean", "bad"), ("bad", "clean")])
@pytest.mark.parametrize("T,k,E", [(4096, 8, 256), (300, 8, 2048), (64, 8, 256), (1, 1, 1)],
                         ids=["cluster_path", "three_kernel_path", "one_cta_path", "one_slot"])
def test_noalloc_matches_oracle_on_two_calls_in_a_row(T, k, E, order):
    build()
    rng = np.random.Generator(np.random.PCG64(T + E + len(order[0])))
    # two calls in a row with different inputs on the one scratch; an invalid
    # id's flag must come through, and the call after it must report clean
    for call, kind in enumerate(order, 1):
        bad = kind == "bad" and T > 1
        flag = _check_one_call(_ids(rng, T, k, E, bad=bad), E, f"{kind} call {call}")
        assert (flag != 0) == bad, f"{kind} call {call}: flag {flag}"


def test_noalloc_sequence_of_sizes_and_paths_on_one_scratch():
    # a large three-kernel build fills most of the scratch with per-chunk
    # histograms; smaller builds on every path follow it, and each must match
    # the oracle exactly
    build()
    rng = np.random.Generator(np.random.PCG64(4242))
    seq = [(100000, 8, 256, True), (40000, 8, 256, False), (300, 8, 2048, False), (4096, 8, 256, True),
           (1, 1, 1, False), (64, 8, 256, False), (100000, 8, 256, False), (7, 3, 5, True)]
    for i, (T, k, E, bad) in enumerate(seq):
        assert nqg.moe_build_row_map_workspace_size(T, k, E) <= (1 << 20)
        flag = _check_one_call(_ids(rng, T, k, E, bad=bad), E, f"step {i}: T={T} k={k} E={E}")
        assert (flag != 0) == bad


def test_noalloc_rejects_problems_beyond_its_scratch():
    build()
    T, k, E = 4096, 8, 8192  # needs a workspace just over the 1 MiB scratch
    assert nqg.moe_build_row_map_workspace_size(T, k, E) > (1 << 20)
    ids = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    counts, offsets, row_map, src_row = _outputs(T, k, E)
    st = nqg.lib().moe_build_row_map_noalloc(
        C.c_void_p(ids.data_ptr()), T, k, E, C.c_void_p(counts.data_ptr()), C.c_void_p(offsets.data_ptr()),
        C.c_void_p(row_map.data_ptr()), None, None, C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == nqg.MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(counts == -9)  # nothing was launched
