"""CPU oracle for TopK selection -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (``topk_selection_gb300``)
never does, and the two share no code.

``oracle.cc`` holds the definitions (plain single-threaded C++17: std::sort
descending for int32; std::stable_sort of column indices for rows, so the
lower index wins among equal values) and an exact one-pass checker for int32
results at sizes where a full sort is too slow.  Each function cites the page
section it follows; the tests pin each against brute force, hand-worked
fixtures, closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_DIR = os.path.join(_HERE, "_lib")
_SRC = os.path.join(_HERE, "oracle.cc")
_lock = threading.Lock()
_libs: dict = {}

# Deliberately wrong variants, built only by the tests that show the pins
# reject them.  The plain build defines none of these.
PLANTED = ("ORACLE_PLANT_ASCENDING", "ORACLE_PLANT_DEDUP", "ORACLE_PLANT_UNSTABLE",
           "ORACLE_PLANT_NAN_LOW", "ORACLE_PLANT_SIGNED_ZERO", "ORACLE_PLANT_SUM_WRAP", "ORACLE_PLANT_ZERO_ORDER",
           "ORACLE_PLANT_KEEP_IGNORED", "ORACLE_PLANT_SORT_UNSTABLE", "ORACLE_PLANT_U32_SIGNED",
           "ORACLE_PLANT_F32_SIGNED_BITS", "ORACLE_PLANT_NAN_PAYLOAD")


def _lib_path(plant):
    return os.path.join(_LIB_DIR, "liboracle.so" if plant is None else f"liboracle_{plant.lower()}.so")


def build(plant: str | None = None, force: bool = False) -> str:
    """Compile oracle.cc with g++ -O2 (one translation unit, a second or two)."""
    if plant is not None and plant not in PLANTED:
        raise ValueError(plant)
    path = _lib_path(plant)
    if not force and os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return path
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-o", tmp, _SRC]
    if plant is not None:
        cmd.insert(1, f"-D{plant}=1")
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


_FAST_SRC = os.path.join(_HERE, "cpu_fast.cc")
_FAST_PATH = os.path.join(_LIB_DIR, "libcpu_fast.so")
_fast_lib = None


def build_fast(force: bool = False) -> str:
    """Compile cpu_fast.cc, the multi-threaded CPU baseline (not an oracle)."""
    if not force and os.path.exists(_FAST_PATH) and os.path.getmtime(_FAST_PATH) >= os.path.getmtime(_FAST_SRC):
        return _FAST_PATH
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _FAST_PATH + f".tmp{os.getpid()}"
    subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-o", tmp, _FAST_SRC], check=True)
    os.replace(tmp, _FAST_PATH)
    return _FAST_PATH


def fast_topk_i32(x, k: int, threads: int = 0):
    """The fast CPU baseline (cpu_fast.cc): per-thread std::nth_element over
    contiguous chunks, then a merge.  Returns (top-k descending, threads
    used).  Timed by bench.py beside the oracle; never used as a check."""
    global _fast_lib
    with _lock:
        if _fast_lib is None:
            lib = ctypes.CDLL(build_fast())
            lib.cpu_fast_topk_i32.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_int]
            lib.cpu_fast_topk_i32.restype = ctypes.c_int
            lib.cpu_fast_hardware_threads.argtypes = []
            lib.cpu_fast_hardware_threads.restype = ctypes.c_int
            _fast_lib = lib
    a = np.ascontiguousarray(x, dtype=np.int32).reshape(-1)
    out = np.empty(max(k, 0), dtype=np.int32)
    used = _fast_lib.cpu_fast_topk_i32(a.ctypes.data, a.size, int(k), out.ctypes.data, int(threads))
    if used < 0:
        raise OracleError(f"cpu_fast_topk_i32 rejected n={a.size} k={k}")
    return out, int(used)


def hardware_threads() -> int:
    """std::thread::hardware_concurrency() of this host."""
    fast_topk_i32(np.zeros(1, np.int32), 1)  # loads the library
    return int(_fast_lib.cpu_fast_hardware_threads())


def load(plant: str | None = None):
    with _lock:
        lib = _libs.get(plant)
        if lib is None:
            lib = ctypes.CDLL(build(plant))
            vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
            lib.oracle_topk_i32.argtypes = [vp, sz, ci, vp]
            lib.oracle_topk_i32.restype = ci
            lib.oracle_topk_rows_f32.argtypes = [vp, ci, ci, ci, vp, vp]
            lib.oracle_topk_rows_f32.restype = ci
            lib.oracle_check_topk_i32.argtypes = [vp, sz, ci, vp]
            lib.oracle_check_topk_i32.restype = ci
            lib.oracle_reduce_i32.argtypes = [vp, sz, ci, vp]
            lib.oracle_reduce_i32.restype = ci
            lib.oracle_reduce_f32.argtypes = [vp, sz, ci, vp]
            lib.oracle_reduce_f32.restype = ci
            lib.oracle_topk_items_f32.argtypes = [vp, vp, vp, sz, ci, vp, vp, vp]
            lib.oracle_topk_items_f32.restype = ci
            lib.oracle_sort_u32.argtypes = [vp, vp, sz, vp, vp]
            lib.oracle_sort_u32.restype = ci
            lib.oracle_topk_u32.argtypes = [vp, sz, ci, vp]
            lib.oracle_topk_u32.restype = ci
            lib.oracle_topk_f32.argtypes = [vp, sz, ci, vp]
            lib.oracle_topk_f32.restype = ci
            _libs[plant] = lib
    return lib


class OracleError(ValueError):
    pass


def topk_i32(x, k: int, plant: str | None = None) -> np.ndarray:
    """The k largest values of int32 array ``x``, sorted descending."""
    a = np.ascontiguousarray(x, dtype=np.int32).reshape(-1)
    out = np.empty(max(k, 0), dtype=np.int32)
    rc = load(plant).oracle_topk_i32(a.ctypes.data, a.size, int(k), out.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle_topk_i32 rejected n={a.size} k={k}")
    return out


def topk_u32(x, k: int, plant: str | None = None) -> np.ndarray:
    """The k largest values of uint32 array ``x``, sorted descending."""
    a = np.ascontiguousarray(x, dtype=np.uint32).reshape(-1)
    out = np.empty(max(k, 0), dtype=np.uint32)
    rc = load(plant).oracle_topk_u32(a.ctypes.data, a.size, int(k), out.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle_topk_u32 rejected n={a.size} k={k}")
    return out


def topk_f32(x, k: int, plant: str | None = None) -> np.ndarray:
    """The k largest values of float32 array ``x`` under IEEE 754 totalOrder,
    sorted descending (bits copied; -0 below +0, NaNs by sign and payload)."""
    a = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(max(k, 0), dtype=np.float32)
    rc = load(plant).oracle_topk_f32(a.ctypes.data, a.size, int(k), out.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle_topk_f32 rejected n={a.size} k={k}")
    return out


def topk_rows_f32(x, k: int, plant: str | None = None):
    """Per-row TopK of a 2-D float32 array: (values, column indices), rows x k."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    if a.ndim != 2:
        raise OracleError("rows input must be 2-D")
    rows, cols = a.shape
    vals = np.empty((rows, max(k, 0)), dtype=np.float32)
    idx = np.empty((rows, max(k, 0)), dtype=np.int32)
    rc = load(plant).oracle_topk_rows_f32(a.ctypes.data, rows, cols, int(k), vals.ctypes.data, idx.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle_topk_rows_f32 rejected rows={rows} cols={cols} k={k}")
    return vals, idx


def check_topk_i32(x, k: int, out) -> bool:
    """True when ``out`` is exactly the TopK of ``x`` (one pass; any size)."""
    a = np.ascontiguousarray(x, dtype=np.int32).reshape(-1)
    o = np.ascontiguousarray(out, dtype=np.int32).reshape(-1)
    if o.size != k:
        return False
    rc = load().oracle_check_topk_i32(a.ctypes.data, a.size, int(k), o.ctypes.data)
    if rc < 0:
        raise OracleError(f"oracle_check_topk_i32 rejected n={a.size} k={k}")
    return rc == 1


REDUCE_OPS = {"sum": 0, "max": 1, "min": 2}


def reduce_i32(x, op: str, plant: str | None = None) -> int:
    """Sum (exact, int64), max or min of an int32 array."""
    a = np.ascontiguousarray(x, dtype=np.int32).reshape(-1)
    out = np.zeros(1, dtype=np.int64)
    rc = load(plant).oracle_reduce_i32(a.ctypes.data, a.size, REDUCE_OPS[op], out.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle_reduce_i32 rejected n={a.size} op={op}")
    return int(out[0])


def reduce_f32(x, op: str, plant: str | None = None) -> float:
    """Sum (left to right in double), max or min (NaN if any NaN; -0 below
    +0) of a float32 array, as a Python float (a double)."""
    a = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.zeros(1, dtype=np.float64)
    rc = load(plant).oracle_reduce_f32(a.ctypes.data, a.size, REDUCE_OPS[op], out.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle_reduce_f32 rejected n={a.size} op={op}")
    return float(out[0])


def topk_items_f32(score, k: int, item=None, keep=None, plant: str | None = None):
    """Score-keyed TopK with item ids and an optional filter: (scores, items,
    count); see oracle_topk_items_f32."""
    sc = np.ascontiguousarray(score, dtype=np.float32).reshape(-1)
    it = None if item is None else np.ascontiguousarray(item, dtype=np.int64).reshape(-1)
    kp = None if keep is None else np.ascontiguousarray(keep, dtype=np.uint8).reshape(-1)
    if it is not None and it.size != sc.size or kp is not None and kp.size != sc.size:
        raise OracleError("item and keep must match score in size")
    os_ = np.empty(max(k, 0), dtype=np.float32)
    oi = np.empty(max(k, 0), dtype=np.int64)
    cnt = np.zeros(1, dtype=np.int64)
    rc = load(plant).oracle_topk_items_f32(sc.ctypes.data, None if it is None else it.ctypes.data,
                                           None if kp is None else kp.ctypes.data, sc.size, int(k),
                                           os_.ctypes.data, oi.ctypes.data, cnt.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle_topk_items_f32 rejected n={sc.size} k={k}")
    return os_, oi, int(cnt[0])


def sort_u32(keys, vals=None, plant: str | None = None):
    """Stable ascending sort of uint32 keys, carrying uint32 values if given:
    (keys, values or None)."""
    k = np.ascontiguousarray(keys, dtype=np.uint32).reshape(-1)
    v = None if vals is None else np.ascontiguousarray(vals, dtype=np.uint32).reshape(-1)
    if v is not None and v.size != k.size:
        raise OracleError("vals must match keys")
    ko = np.empty_like(k)
    vo = None if v is None else np.empty_like(v)
    rc = load(plant).oracle_sort_u32(k.ctypes.data, None if v is None else v.ctypes.data, k.size, ko.ctypes.data,
                                     None if vo is None else vo.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle_sort_u32 rejected n={k.size}")
    return ko, vo
