"""The workspace-free routing build, for callers that cannot allocate device
memory (framework plug-ins that own no memory of their own, loops that may
not call cudaMalloc).  Called through the C ABI, it must give exactly what
the regular entry point gives, call after call, although every call reuses
the library's one fixed scratch array.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""
import ctypes as C

import numpy as np
import pytest
import torch

import norm_quant_gb300 as nqg
from norm_quant_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ids(rng, T, k, E, bad=False):
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, k)) < 0.1] = -1
    if bad:
        ids[T // 2, 0] = E + 3
    return torch.from_numpy(ids).to(DEV)


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
    """The new entry point, called through ctypes with raw device pointers."""
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


@pytest.mark.parametrize("T,k,E", [(4096, 8, 256), (300, 8, 2048), (1, 1, 1)],
                         ids=["cluster_path", "three_kernel_path", "one_slot"])
def test_noalloc_matches_regular_on_two_calls_in_a_row(T, k, E):
    build()
    rng = np.random.Generator(np.random.PCG64(T + E))
    # two calls in a row with different inputs: the second must not see
    # anything the first left in the shared scratch (the second also holds an
    # invalid id, whose flag must come through)
    for call, bad in ((1, False), (2, T > 1)):
        ids = _ids(rng, T, k, E, bad=bad)
        c0, o0, r0, s0, st0 = _regular(ids, E)
        c1, o1, r1, s1, flag = _noalloc(ids, E)
        assert torch.equal(c0, c1) and torch.equal(o0, o1) and torch.equal(r0, r1), f"call {call}"
        n_valid = int(o0[E].item())
        assert torch.equal(s0[:n_valid], s1[:n_valid]), f"call {call}"
        assert (flag != 0) == (st0 == nqg.MOE_ERR_INVALID_EXPERT) == bad, f"call {call}"


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
