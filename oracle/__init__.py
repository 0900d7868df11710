"""CPU oracle for the MoE combine/finalize step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product path
(``norm_quant_gb300``) never touches it, and it never touches the product
path: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, fp64, fixed order); this
module compiles it with gcc on first use and marshals numpy arrays into it.
bf16 arrays are passed as their raw ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

QUANT = {None: 0, "none": 0, "mxfp8": 1, "nvfp4": 2, "mxfp4": 3}
IO_DTYPE = {"bf16": 0, "fp16": 1}
WEIGHT_DTYPE = {"fp32": 0, "bf16": 1, "fp16": 2}
LAYOUT = {"linear": 0, "swizzled": 1, "128x4": 1}


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, no fast-math,
    no FMA contraction, so x86 and Arm hosts give identical results)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_OUT_DIR)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class CombineArgs(C.Structure):
    _fields_ = [
        ("T", C.c_int64), ("H", C.c_int32), ("k", C.c_int32),
        ("expert_out", C.c_void_p), ("n_rows", C.c_int64),
        ("row_map", C.c_void_p), ("weights", C.c_void_p),
        ("shared", C.c_void_p), ("residual", C.c_void_p), ("gamma", C.c_void_p),
        ("eps", C.c_float), ("weight_bias", C.c_float),
        ("quant", C.c_int32), ("sf_layout", C.c_int32), ("global_scale", C.c_float),
        ("combined_out", C.c_void_p), ("residual_out", C.c_void_p),
        ("norm_out", C.c_void_p), ("quant_out", C.c_void_p),
        ("scales_out", C.c_void_p), ("y_out", C.c_void_p),
        ("expert_layout", C.c_int32), ("io_dtype", C.c_int32), ("weight_dtype", C.c_int32),
        ("pad0", C.c_int32),
    ]


def lib() -> C.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            L.oracle_bf16_to_f64.restype = C.c_double
            L.oracle_bf16_to_f64.argtypes = [C.c_uint16]
            L.oracle_f64_to_bf16.restype = C.c_uint16
            L.oracle_f64_to_bf16.argtypes = [C.c_double]
            L.oracle_f16_to_f64.restype = C.c_double
            L.oracle_f16_to_f64.argtypes = [C.c_uint16]
            L.oracle_f64_to_f16.restype = C.c_uint16
            L.oracle_f64_to_f16.argtypes = [C.c_double]
            L.oracle_ue8m0_fp4_for_amax.restype = C.c_uint8
            L.oracle_ue8m0_fp4_for_amax.argtypes = [C.c_double]
            L.oracle_dequant_mxfp4.restype = None
            L.oracle_dequant_mxfp4.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int32,
                                               C.c_int32, C.c_void_p]
            L.oracle_e4m3_to_f64.restype = C.c_double
            L.oracle_e4m3_to_f64.argtypes = [C.c_uint8]
            L.oracle_e4m3_from_f64.restype = C.c_uint8
            L.oracle_e4m3_from_f64.argtypes = [C.c_double]
            L.oracle_e2m1_to_f64.restype = C.c_double
            L.oracle_e2m1_to_f64.argtypes = [C.c_uint8]
            L.oracle_e2m1_from_f64.restype = C.c_uint8
            L.oracle_e2m1_from_f64.argtypes = [C.c_double]
            L.oracle_ue8m0_for_amax.restype = C.c_uint8
            L.oracle_ue8m0_for_amax.argtypes = [C.c_double]
            L.oracle_sf_offset.restype = C.c_int64
            L.oracle_sf_offset.argtypes = [C.c_int64, C.c_int64, C.c_int64, C.c_int32]
            L.oracle_sf_offsets.restype = None
            L.oracle_sf_offsets.argtypes = [C.c_int64, C.c_int64, C.c_int32, C.c_void_p]
            L.oracle_scales_bytes.restype = C.c_int64
            L.oracle_scales_bytes.argtypes = [C.c_int64, C.c_int32, C.c_int32, C.c_int32]
            L.oracle_build_row_map.restype = C.c_int
            L.oracle_build_row_map.argtypes = [C.c_void_p, C.c_int64, C.c_int32, C.c_int32,
                                               C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
            L.oracle_combine_args_size.restype = C.c_int
            L.oracle_combine.restype = C.c_int
            L.oracle_combine.argtypes = [C.POINTER(CombineArgs)]
            L.oracle_dispatch_permute.restype = C.c_int
            L.oracle_dispatch_permute.argtypes = [C.c_void_p, C.c_int64, C.c_int32, C.c_void_p,
                                                  C.c_int32, C.c_void_p, C.c_int64]
            L.oracle_dequant_mxfp8.restype = None
            L.oracle_dequant_mxfp8.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int32,
                                               C.c_int32, C.c_void_p]
            L.oracle_dequant_nvfp4.restype = None
            L.oracle_dequant_nvfp4.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int32,
                                               C.c_int32, C.c_float, C.c_void_p]
            assert L.oracle_combine_args_size() == C.sizeof(CombineArgs)
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats --

def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    f = lib().oracle_f64_to_bf16
    x = np.asarray(x, dtype=np.float64)
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


_F16_TABLE = None


def f16_to_f64(bits) -> np.ndarray:
    global _F16_TABLE
    if _F16_TABLE is None:
        f = lib().oracle_f16_to_f64
        _F16_TABLE = np.array([f(i) for i in range(1 << 16)], dtype=np.float64)
    return _F16_TABLE[np.asarray(bits, dtype=np.uint16)]


def f64_to_f16(x) -> np.ndarray:
    f = lib().oracle_f64_to_f16
    x = np.asarray(x, dtype=np.float64)
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def ue8m0_fp4_for_amax(amax) -> np.ndarray:
    f = lib().oracle_ue8m0_fp4_for_amax
    a = np.asarray(amax, dtype=np.float64)
    return np.array([f(float(v)) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def e4m3_to_f64(codes) -> np.ndarray:
    f = lib().oracle_e4m3_to_f64
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([f(i) for i in range(256)], dtype=np.float64)
    return table[c]


def e4m3_from_f64(x) -> np.ndarray:
    f = lib().oracle_e4m3_from_f64
    x = np.asarray(x, dtype=np.float64)
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint8).reshape(x.shape)


def e2m1_to_f64(codes) -> np.ndarray:
    f = lib().oracle_e2m1_to_f64
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([f(i) for i in range(16)], dtype=np.float64)
    return table[c & 15]


def e2m1_from_f64(x) -> np.ndarray:
    f = lib().oracle_e2m1_from_f64
    x = np.asarray(x, dtype=np.float64)
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint8).reshape(x.shape)


def ue8m0_for_amax(amax) -> np.ndarray:
    f = lib().oracle_ue8m0_for_amax
    a = np.asarray(amax, dtype=np.float64)
    return np.array([f(float(v)) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def sf_offset(r: int, c: int, C_cols: int, layout="linear") -> int:
    return int(lib().oracle_sf_offset(int(r), int(c), int(C_cols), LAYOUT[layout]))


def sf_offsets(T: int, C_cols: int, layout="linear") -> np.ndarray:
    """int64 [T, C_cols] table of sf_offset(r, c)."""
    out = np.zeros((T, C_cols), np.int64)
    lib().oracle_sf_offsets(int(T), int(C_cols), LAYOUT[layout], _ptr(out))
    return out


def scales_bytes(T: int, H: int, quant: str, layout="linear") -> int:
    return int(lib().oracle_scales_bytes(int(T), int(H), QUANT[quant], LAYOUT[layout]))


# ---------------------------------------------------------------- routing --

def build_row_map(topk_ids: np.ndarray, E: int):
    """Returns (status, counts[E], offsets[E+1], row_map[T,k], src_row[N_v])."""
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    row_map = np.zeros((T, k), np.int32)
    src_row = np.full(max(T * k, 1), -1, np.int32)
    st = lib().oracle_build_row_map(_ptr(ids), T, k, E, _ptr(counts), _ptr(offsets),
                                    _ptr(row_map), _ptr(src_row))
    return st, counts, offsets, row_map, src_row[: int(offsets[E])]


# ---------------------------------------------------------------- combine --

def combine(expert_out, row_map, weights, *, shared=None, residual=None, gamma=None,
            eps=1e-6, weight_bias=0.0, quant=None, sf_layout="linear",
            global_scale=1.0, outputs=("combined", "residual", "norm", "quant", "y"),
            expert_layout="grouped", io_dtype="bf16", weight_dtype="fp32"):
    """Run the oracle on host arrays.

    expert_out: uint16 bf16 bits [n_rows, H] grouped by expert (row_map int32
    [T, k]) or, with expert_layout="slot_major", [k, T, H] (row_map unused);
    weights fp32 [T, k]; shared / residual: uint16 [T, H] or None; gamma: uint16 [H]
    or None (no RMSNorm).  Returns a dict with the requested outputs
    (combined / residual / norm as uint16 bf16 or fp16 bits (io_dtype),
    quant + scales as uint8,
    y as the fp64 quantiser input) and 'status'."""
    ex = _c(expert_out, np.uint16)
    w = _c(weights, np.float32 if weight_dtype == "fp32" else np.uint16)
    T, k = w.shape
    slot_major = expert_layout == "slot_major"
    rm = None if slot_major else _c(row_map, np.int32)
    if slot_major:
        ex = ex.reshape(k * T, -1)      # [k, T, H] -> rows j * T + t
    H = ex.shape[1] if ex.ndim == 2 else int(np.asarray(residual if residual is not None
                                                         else shared).shape[1])
    sh = _c(shared, np.uint16)
    rs = _c(residual, np.uint16)
    gm = _c(gamma, np.uint16)
    out = {}
    if "combined" in outputs:
        out["combined"] = np.zeros((T, H), np.uint16)
    if "residual" in outputs:
        out["residual"] = np.zeros((T, H), np.uint16)
    if "norm" in outputs and gm is not None:
        out["norm"] = np.zeros((T, H), np.uint16)
    qk = QUANT[quant]
    if qk and "quant" in outputs:
        out["quant"] = np.zeros((T, H if qk == 1 else H // 2), np.uint8)  # fp4: 2 per byte
        out["scales"] = np.zeros(scales_bytes(T, H, quant, sf_layout), np.uint8)
    if "y" in outputs:
        out["y"] = np.zeros((T, H), np.float64)
    a = CombineArgs(
        T=T, H=H, k=k, expert_out=_ptr(ex), n_rows=(ex.shape[0] if ex.ndim == 2 else 0),
        row_map=_ptr(rm), weights=_ptr(w), shared=_ptr(sh), residual=_ptr(rs),
        gamma=_ptr(gm), eps=eps, weight_bias=weight_bias, quant=qk,
        sf_layout=LAYOUT[sf_layout], global_scale=global_scale,
        combined_out=_ptr(out.get("combined")), residual_out=_ptr(out.get("residual")),
        norm_out=_ptr(out.get("norm")), quant_out=_ptr(out.get("quant")),
        scales_out=_ptr(out.get("scales")), y_out=_ptr(out.get("y")),
        expert_layout=1 if slot_major else 0, io_dtype=IO_DTYPE[io_dtype],
        weight_dtype=WEIGHT_DTYPE[weight_dtype])
    out["status"] = lib().oracle_combine(C.byref(a))
    return out


def dispatch_permute(x: np.ndarray, row_map: np.ndarray, n_rows: int, fill: int = 0):
    """x_grouped [n_rows, H] (uint16 bf16 bits) with x[t] copied to every row
    row_map[t, j] >= 0; other rows hold `fill`.  Returns (status, x_grouped)."""
    xx = _c(x, np.uint16)
    rm = _c(row_map, np.int32)
    T, H = xx.shape
    out = np.full((n_rows, H), fill, np.uint16)
    st = lib().oracle_dispatch_permute(_ptr(xx), T, H, _ptr(rm), rm.shape[1], _ptr(out), n_rows)
    return st, out


def dequant(q: np.ndarray, scales: np.ndarray, T: int, H: int, quant: str,
            sf_layout="linear", global_scale=1.0) -> np.ndarray:
    """Dequantise codes + scales to fp64 [T, H] by the formats' definitions."""
    q = _c(q, np.uint8)
    s = _c(scales, np.uint8)
    out = np.zeros((T, H), np.float64)
    if QUANT[quant] == 1:
        lib().oracle_dequant_mxfp8(_ptr(q), _ptr(s), T, H, LAYOUT[sf_layout], _ptr(out))
    elif QUANT[quant] == 3:
        lib().oracle_dequant_mxfp4(_ptr(q), _ptr(s), T, H, LAYOUT[sf_layout], _ptr(out))
    else:
        lib().oracle_dequant_nvfp4(_ptr(q), _ptr(s), T, H, LAYOUT[sf_layout],
                                   global_scale, _ptr(out))
    return out
