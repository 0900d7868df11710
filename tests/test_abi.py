"""The C ABI without a GPU: the library builds and loads, exports every
function include/*.h declares, agrees on the argument struct's layout, sizes
workspaces and scale matrices like the oracle, and rejects invalid calls on
the host before anything is launched (these calls never reach CUDA)."""
import ctypes as C
import glob
import os
import re

import pytest

import norm_quant_gb300 as nqg
import oracle
from norm_quant_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build()
    return nqg.lib()


def _declared():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M))
    return names


def test_every_declared_symbol_is_exported(L):
    declared = _declared()
    assert {"moe_build_row_map", "moe_combine", "moe_build_row_map_check"} <= declared
    for name in declared:
        assert hasattr(L, name), name
    assert set(nqg.SYMBOLS) == declared  # the binding declares exactly the header's entry points


def test_abi_version_and_struct(L):
    assert nqg.moe_abi_version() == nqg.ABI_VERSION
    assert L.moe_combine_args_size() == C.sizeof(nqg.MoeCombineArgs) == 152
    assert nqg.moe_status_string(0) == "MOE_OK"
    assert "INVALID_EXPERT" in nqg.moe_status_string(4)


@pytest.mark.parametrize("T,H,q,lay", [(4096, 7168, "mxfp8", "linear"), (8192, 4096, "nvfp4", "swizzled"),
                                       (1, 32, "mxfp8", "swizzled"), (130, 96, "mxfp8", "swizzled"),
                                       (70, 64, "mxfp4", "swizzled"), (9, 96, "mxfp4", "linear"),
                                       (7, 48, "nvfp4", "linear"), (0, 64, "nvfp4", "swizzled")])
def test_scales_bytes_match_oracle(L, T, H, q, lay):
    assert nqg.moe_scales_bytes(T, H, q, lay) == oracle.scales_bytes(T, H, q, lay)


def test_workspace_size_grows_with_slots(L):
    a = nqg.moe_build_row_map_workspace_size(64, 8, 256)
    b = nqg.moe_build_row_map_workspace_size(16384, 8, 256)
    assert 0 < a < b and b % 256 == 0


def _args(**kw):
    base = dict(T=4, H=64, top_k=2, expert_out=0x1000, n_expert_rows=8, row_map=0x2000,
                router_weights=0x3000, shared_out=None, residual=None, gamma=None, eps=1e-6,
                weight_bias=0.0, quant=0, sf_layout=0, global_scale=1.0, expert_layout=0,
                combined_out=0x4000, residual_out=None, norm_out=None, quant_out=None,
                scales_out=None, status=None)
    base.update(kw)
    return nqg.MoeCombineArgs(**base)


@pytest.mark.parametrize("kw,want", [
    (dict(H=60), 1), (dict(H=0), 1), (dict(H=32768), 2), (dict(top_k=0), 1), (dict(top_k=33), 2),
    (dict(T=-1), 1), (dict(row_map=None), 1), (dict(router_weights=None), 1),
    (dict(expert_out=None), 1), (dict(combined_out=None), 1), (dict(quant=3), 1),
    (dict(quant=1, H=48, quant_out=0x5000, scales_out=0x6000), 1),
    (dict(quant=1), 1), (dict(quant=2, quant_out=0x5000, scales_out=0x6000, global_scale=0.0), 1),
    (dict(quant=2, quant_out=0x5000, scales_out=0x6000, global_scale=float("inf")), 1),
    (dict(quant=1, quant_out=0x5000, scales_out=0x6000, sf_layout=2), 1),
    (dict(norm_out=0x7000), 1), (dict(expert_out=0x1008), 1), (dict(combined_out=0x4004), 1),
    (dict(row_map=0x2002), 1), (dict(eps=-1.0), 1), (dict(eps=float("nan")), 1),
    (dict(expert_layout=2), 1), (dict(status=0x8002), 1),
    (dict(io_dtype=2), 1), (dict(weight_dtype=3), 1), (dict(router_weights=0x3002), 1),
    (dict(quant=3, H=48, quant_out=0x5000, scales_out=0x6000), 1),  # MXFP4 needs H % 32
    (dict(expert_layout=1, row_map=None, n_expert_rows=7), 1),  # slot-major needs top_k * T rows
    (dict(T=0), 0),  # a valid no-op: returns before any CUDA call
    (dict(T=0, row_map=None, router_weights=None, expert_out=None, combined_out=None), 0),
])
def test_combine_validation(L, kw, want):
    a = _args(**kw)
    assert L.moe_combine(C.byref(a), None) == want


def test_tuning_validation(L):
    assert L.moe_tuning_set(3, 0, 0, 0, 0, 0) == 1
    assert L.moe_tuning_set(0, 13, 0, 0, 0, 0) == 1
    assert L.moe_tuning_set(0, 0, 300, 0, 0, 0) == 1
    assert L.moe_tuning_set(0, 0, 0, 9, 0, 0) == 1
    assert L.moe_tuning_set(0, 0, 0, 0, 17, 0) == 1
    assert L.moe_tuning_set(0, 0, 0, 0, -2, 0) == 1
    for bad in (-1, 3, 6, 32):
        assert L.moe_tuning_set(0, 0, 0, 0, 0, bad) == 1
    assert L.moe_tuning_set(2, 2, 144, 1, -1, 8) == 0
    assert L.moe_tuning_set(0, 0, 0, 0, 0, 0) == 0
    assert L.moe_debug_stall(-2) == 1
    assert L.moe_debug_stall(-1) == 0


def test_combine_null_args(L):
    assert L.moe_combine(None, None) == 1


def test_route_validation(L):
    n = C.c_size_t(0)
    assert L.moe_build_row_map_workspace_size(10, 0, 8, C.byref(n)) == 1
    assert L.moe_build_row_map_workspace_size(10, 33, 8, C.byref(n)) == 2
    assert L.moe_build_row_map_workspace_size(10, 4, 9000, C.byref(n)) == 2
    assert L.moe_build_row_map_workspace_size(1 << 29, 8, 8, C.byref(n)) == 2
    ws = 0x10000
    # T > 0 with a NULL ids / row_map pointer, misaligned workspace, too small workspace
    assert L.moe_build_row_map(None, 4, 2, 8, 0x100, 0x200, 0x300, None, ws, 1 << 20, None) == 1
    assert L.moe_build_row_map(0x400, 4, 2, 8, 0x100, 0x200, None, None, ws, 1 << 20, None) == 1
    assert L.moe_build_row_map(0x400, 4, 2, 8, 0x100, 0x200, 0x300, None, ws + 4, 1 << 20, None) == 1
    assert L.moe_build_row_map(0x400, 4, 2, 8, 0x100, 0x200, 0x300, None, ws, 8, None) == 3
    assert L.moe_build_row_map(0x400, 4, 2, 8, 0x100, 0x200, 0x300, None, None, 0, None) == 3
    assert L.moe_build_row_map(0x400, 4, 2, 8, None, 0x200, 0x300, None, ws, 1 << 20, None) == 1
    k = C.c_int32(-1)
    assert L.moe_build_row_map_launches(10, 4, 8, None) == 1
    assert L.moe_build_row_map_launches(-1, 4, 8, C.byref(k)) == 1
    assert L.moe_build_row_map_launches(10, 33, 8, C.byref(k)) == 2
    assert L.moe_build_row_map_launches(0, 4, 8, C.byref(k)) == 0 and k.value == 0


def test_dispatch_validation(L):
    assert L.moe_dispatch_permute(0x1000, 4, 60, 0x2000, 2, 0x3000, 8, None, None) == 1   # H % 8
    assert L.moe_dispatch_permute(0x1000, 4, 32768, 0x2000, 2, 0x3000, 8, None, None) == 2
    assert L.moe_dispatch_permute(0x1000, 4, 64, 0x2000, 0, 0x3000, 8, None, None) == 1   # top_k
    assert L.moe_dispatch_permute(None, 4, 64, 0x2000, 2, 0x3000, 8, None, None) == 1
    assert L.moe_dispatch_permute(0x1008, 4, 64, 0x2000, 2, 0x3000, 8, None, None) == 1   # alignment
    assert L.moe_dispatch_permute(0x1000, 4, 64, 0x2002, 2, 0x3000, 8, None, None) == 1
    assert L.moe_dispatch_permute(None, 0, 64, None, 2, None, 0, None, None) == 0          # empty batch
