"""MoE combine/finalize on one GB300 -- Python binding of ``libnqg.so``.

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (torch provides device memory
and streams); bf16 tensors may be ``torch.bfloat16`` or raw 16-bit views.
The entry points have the names of the C ABI in ``include/moe_combine.h``.

There is no fallback: if the library is not built, every call raises.
Build it with ``norm_quant_gb300.build.build()`` (``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes as C
import os
import threading

from .build import LIB_PATH, build  # noqa: F401  (re-exported)

QUANT = {None: 0, "none": 0, "mxfp8": 1, "nvfp4": 2, "mxfp4": 3}
IO_DTYPE = {"bf16": 0, "fp16": 1}
WEIGHT_DTYPE = {"fp32": 0, "bf16": 1, "fp16": 2}
LAYOUT = {"linear": 0, "swizzled": 1, "128x4": 1}
EXPERT_LAYOUT = {"grouped": 0, "slot_major": 1}
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_INVALID_EXPERT = 4
MOE_ERR_CUDA = 5
MOE_ERR_ROW_OUT_OF_RANGE = 6
MOE_ERR_DEVICE_TIMEOUT = 7
ABI_VERSION = 4


class MoeCombineArgs(C.Structure):
    """Mirror of ``moe_combine_args`` (include/moe_combine.h)."""
    _fields_ = [
        ("T", C.c_int64), ("H", C.c_int32), ("top_k", C.c_int32),
        ("expert_out", C.c_void_p), ("n_expert_rows", C.c_int64),
        ("row_map", C.c_void_p), ("router_weights", C.c_void_p),
        ("shared_out", C.c_void_p), ("residual", C.c_void_p), ("gamma", C.c_void_p),
        ("eps", C.c_float), ("weight_bias", C.c_float),
        ("quant", C.c_int32), ("sf_layout", C.c_int32), ("global_scale", C.c_float),
        ("expert_layout", C.c_int32),
        ("combined_out", C.c_void_p), ("residual_out", C.c_void_p), ("norm_out", C.c_void_p),
        ("quant_out", C.c_void_p), ("scales_out", C.c_void_p), ("status", C.c_void_p),
        ("io_dtype", C.c_int32), ("weight_dtype", C.c_int32),
    ]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {moe_status_string(status)} ({status})")
        self.status = status


_lock = threading.Lock()
_lib = None

# C symbols declared in include/moe_combine.h, with (restype, argtypes).
SYMBOLS = {
    "moe_abi_version": (C.c_int, []),
    "moe_status_string": (C.c_char_p, [C.c_int]),
    "moe_combine_args_size": (C.c_size_t, []),
    "moe_build_row_map_workspace_size": (C.c_int, [C.c_int64, C.c_int32, C.c_int32,
                                                   C.POINTER(C.c_size_t)]),
    "moe_build_row_map": (C.c_int, [C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_void_p,
                                    C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t,
                                    C.c_void_p]),
    "moe_build_row_map_check": (C.c_int, [C.c_void_p, C.c_void_p]),
    "moe_build_row_map_launches": (C.c_int, [C.c_int64, C.c_int32, C.c_int32, C.POINTER(C.c_int32)]),
    "moe_build_row_map_noalloc": (C.c_int, [C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_void_p,
                                            C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "moe_combine": (C.c_int, [C.POINTER(MoeCombineArgs), C.c_void_p]),
    "moe_scales_bytes": (C.c_int, [C.c_int64, C.c_int32, C.c_int32, C.c_int32,
                                   C.POINTER(C.c_size_t)]),
    "moe_tuning_set": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32]),
    "moe_debug_stall": (C.c_int, [C.c_int64]),
    "moe_dispatch_permute": (C.c_int, [C.c_void_p, C.c_int64, C.c_int32, C.c_void_p, C.c_int32,
                                       C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p]),
}


def lib() -> C.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "norm_quant_gb300.build.build() (no fallback path exists)")
            L = C.CDLL(LIB_PATH)
            for name, (res, args) in SYMBOLS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            if L.moe_abi_version() != ABI_VERSION:
                raise RuntimeError("libnqg.so ABI version mismatch")
            if L.moe_combine_args_size() != C.sizeof(MoeCombineArgs):
                raise RuntimeError("moe_combine_args layout mismatch")
            _lib = L
    return _lib


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def moe_abi_version() -> int:
    return int(lib().moe_abi_version())


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _need(t, nbytes: int, name: str):
    """Raises ValueError if tensor t (when given) holds fewer than nbytes
    bytes: the kernels take plain pointers and would read or write past a
    buffer that is too small."""
    if t is not None and t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes; this call needs {nbytes}")


def _scales_bytes(T: int, H: int, vec: int, sf_layout: str) -> int:
    """Bytes of a scale matrix: linear T x C, or 128x4 with rows padded to
    128 and columns to 4 (the library's moe_scales_bytes)."""
    cols = H // vec
    if sf_layout == "linear":
        return T * cols
    return -(-T // 128) * 128 * (-(-cols // 4) * 4)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _check(st: int, what: str):
    if st != MOE_OK:
        raise MoeError(st, what)


def moe_build_row_map_workspace_size(T: int, top_k: int, E: int) -> int:
    n = C.c_size_t(0)
    _check(lib().moe_build_row_map_workspace_size(T, top_k, E, C.byref(n)),
           "moe_build_row_map_workspace_size")
    return n.value


def moe_build_row_map(topk_ids, E: int, counts, offsets, row_map, src_row=None,
                      workspace=None, stream=None) -> None:
    """topk_ids int32 [T, k] -> counts [E], offsets [E+1], row_map [T, k],
    src_row [>= N_valid] (optional).  workspace: uint8 CUDA tensor of at least
    moe_build_row_map_workspace_size(T, k, E) bytes."""
    T, k = topk_ids.shape
    _need(topk_ids, T * k * 4, "topk_ids")
    _need(counts, E * 4, "counts")
    _need(offsets, (E + 1) * 4, "offsets")
    _need(row_map, T * k * 4, "row_map")
    _check(lib().moe_build_row_map(_ptr(topk_ids), T, k, E, _ptr(counts), _ptr(offsets),
                                   _ptr(row_map), _ptr(src_row), _ptr(workspace),
                                   workspace.numel() * workspace.element_size() if workspace is not None else 0,
                                   _stream(stream)),
           "moe_build_row_map")


def moe_build_row_map_noalloc(topk_ids, E: int, counts, offsets, row_map, src_row=None,
                              error_flag=None, stream=None) -> None:
    """moe_build_row_map without a workspace, for callers that cannot
    allocate device memory: the library's own fixed scratch array is used
    (see include/moe_combine.h for its size limit and sharing rules)."""
    T, k = topk_ids.shape
    _need(topk_ids, T * k * 4, "topk_ids")
    _need(counts, E * 4, "counts")
    _need(offsets, (E + 1) * 4, "offsets")
    _need(row_map, T * k * 4, "row_map")
    _need(error_flag, 4, "error_flag")
    _check(lib().moe_build_row_map_noalloc(_ptr(topk_ids), T, k, E, _ptr(counts), _ptr(offsets),
                                           _ptr(row_map), _ptr(src_row), _ptr(error_flag), _stream(stream)),
           "moe_build_row_map_noalloc")


def moe_build_row_map_check(workspace, stream=None) -> int:
    """Synchronises the stream; MOE_OK or MOE_ERR_INVALID_EXPERT."""
    return int(lib().moe_build_row_map_check(_ptr(workspace), _stream(stream)))


def moe_build_row_map_launches(T: int, top_k: int, E: int) -> int:
    """Kernels moe_build_row_map launches for this shape on the current device (1, 3, or 0)."""
    n = C.c_int32(-1)
    _check(lib().moe_build_row_map_launches(T, top_k, E, C.byref(n)), "moe_build_row_map_launches")
    return n.value


def moe_scales_bytes(T: int, H: int, quant: str, sf_layout: str = "linear") -> int:
    n = C.c_size_t(0)
    _check(lib().moe_scales_bytes(T, H, QUANT[quant], LAYOUT[sf_layout], C.byref(n)), "moe_scales_bytes")
    return n.value


def moe_dispatch_permute(x, row_map, x_grouped, status=None, stream=None) -> None:
    """x [T, H] bf16 -> x_grouped [n_rows, H]: row row_map[t, j] >= 0 gets x[t]."""
    T, H = x.shape
    _need(x, T * H * 2, "x")
    _need(row_map, T * row_map.shape[1] * 4, "row_map")
    _need(status, 4, "status")
    _check(lib().moe_dispatch_permute(_ptr(x), T, H, _ptr(row_map), row_map.shape[1], _ptr(x_grouped),
                                      int(x_grouped.shape[0]), _ptr(status), _stream(stream)),
           "moe_dispatch_permute")


def moe_tuning_set(vpt: int = 0, rows_per_slot: int = 0, ring_kib: int = 0, ctas_per_sm: int = 0,
                   route_cluster: int = 0, combine_split: int = 0) -> None:
    """Overrides the launch plans (0 = automatic); results do not depend on it."""
    _check(lib().moe_tuning_set(vpt, rows_per_slot, ring_kib, ctas_per_sm, route_cluster, combine_split),
           "moe_tuning_set")


def moe_debug_stall(slots: int = -1) -> None:
    """Test hook: the combine's CTA 0 stops staging rows after `slots` ring
    slots, so its bounded waits run out and the status reports a timeout
    (-1 turns it off)."""
    _check(lib().moe_debug_stall(slots), "moe_debug_stall")


def combine_args(*, expert_out, row_map, router_weights, shared_out=None, residual=None,
                 gamma=None, eps=1e-6, weight_bias=0.0, quant=None, sf_layout="linear",
                 global_scale=1.0, combined_out=None, residual_out=None, norm_out=None,
                 quant_out=None, scales_out=None, status=None, H=None,
                 expert_layout="grouped", io_dtype="bf16", weight_dtype="fp32") -> MoeCombineArgs:
    """Fills a MoeCombineArgs from tensors (T and top_k from router_weights'
    shape).  expert_layout "slot_major": expert_out is [top_k, T, H] and
    row_map may be None."""
    T, k = router_weights.shape
    if H is None:
        H = int(expert_out.shape[-1])
    n_rows = int(expert_out.numel() // H) if H else 0
    _need(router_weights, T * k * (4 if weight_dtype == "fp32" else 2), "router_weights")
    if expert_layout == "slot_major":
        _need(expert_out, k * T * H * 2, "expert_out")
    else:
        _need(row_map, T * k * 4, "row_map")
    for name, t in (("shared_out", shared_out), ("residual", residual), ("combined_out", combined_out),
                    ("residual_out", residual_out), ("norm_out", norm_out)):
        _need(t, T * H * 2, name)
    _need(gamma, H * 2, "gamma")
    if quant:
        _need(quant_out, T * (H if quant == "mxfp8" else H // 2), "quant_out")
        vec = 16 if quant == "nvfp4" else 32
        if H % vec == 0:  # otherwise the library rejects the call itself
            _need(scales_out, _scales_bytes(T, H, vec, sf_layout), "scales_out")
    _need(status, 4, "status")
    return MoeCombineArgs(
        T=T, H=H, top_k=k, expert_out=_ptr(expert_out), n_expert_rows=n_rows,
        expert_layout=EXPERT_LAYOUT[expert_layout],
        row_map=_ptr(row_map), router_weights=_ptr(router_weights), shared_out=_ptr(shared_out),
        residual=_ptr(residual), gamma=_ptr(gamma), eps=eps, weight_bias=weight_bias,
        quant=QUANT[quant], sf_layout=LAYOUT[sf_layout], global_scale=global_scale,
        combined_out=_ptr(combined_out), residual_out=_ptr(residual_out), norm_out=_ptr(norm_out),
        quant_out=_ptr(quant_out), scales_out=_ptr(scales_out), status=_ptr(status),
        io_dtype=IO_DTYPE[io_dtype], weight_dtype=WEIGHT_DTYPE[weight_dtype])


def moe_combine(stream=None, **kw) -> None:
    """Enqueues the combine; keyword arguments as in combine_args()."""
    args = kw.pop("args", None) or combine_args(**kw)
    _check(lib().moe_combine(C.byref(args), _stream(stream)), "moe_combine")
