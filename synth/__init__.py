"""Seeded synthetic inputs for the TopK workloads (host side, numpy).

This package draws numbers and nothing else: no part of the selection
arithmetic lives here.  Both the CPU oracle (``oracle``) and the CUDA path
(``topk_selection_gb300``) read the arrays it fills, so a parity test always
feeds the two sides the same bytes.

The generator is SplitMix64 evaluated in counter form (``gen.c`` gives the
definition); every workload below names its seed so a run can be repeated.

Workloads, as the TopK pages benchmark them ("CUDA parallel optimisation:
TopK, shared memory and two-stage reduction", section 4.1: 1e7, 1e8 and 1e9
int values, top 20):

* ``i32_uniform(n, seed)``   -- int32 uniform over the full range
* ``i32_ascending(n)``       -- in[i] = i (worst case for a running threshold)
* ``i32_mod(n, seed, m)``    -- int32 uniform in [0, m) (heavy duplicates)
* ``f32_normal(n, seed)``    -- float32 N(0, 1), Box-Muller in double
* ``f32_rows_tied(rows, cols, seed, frac)`` -- N(0,1) rows where
  floor(frac * cols) distinct positions per row are overwritten by copies of
  that row's maximum, so the k-th value of every row is heavily tied
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_DIR = os.path.join(_HERE, "_lib")
_LIB_PATH = os.path.join(_LIB_DIR, "libsynth.so")
_SRC = os.path.join(_HERE, "gen.c")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gen.c`` into ``_lib/libsynth.so`` (plain gcc, -O2)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"],
                   check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, sz, i32p, f32p = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p
            lib.synth_splitmix64_at.restype = u64
            lib.synth_splitmix64_at.argtypes = [u64, u64]
            lib.synth_i32_uniform.argtypes = [i32p, sz, u64, ctypes.c_int]
            lib.synth_i32_mod.argtypes = [i32p, sz, u64, ctypes.c_uint32, ctypes.c_int]
            lib.synth_i32_ascending.argtypes = [i32p, sz, ctypes.c_int]
            lib.synth_f32_normal.argtypes = [f32p, sz, u64, ctypes.c_int]
            lib.synth_f32_force_ties.argtypes = [f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, u64,
                                                 ctypes.c_int]
            for f in ("synth_i32_uniform", "synth_i32_mod", "synth_i32_ascending", "synth_f32_normal",
                      "synth_f32_force_ties"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _threads(nthreads):
    if nthreads is not None:
        return int(nthreads)
    return max(1, min(32, os.cpu_count() or 1))


def _out(out, n, dtype):
    if out is None:
        return np.empty(n, dtype=dtype)
    if out.dtype != dtype or out.size != n or not out.flags.c_contiguous:
        raise ValueError("out must be a contiguous array of the requested size and dtype")
    return out.reshape(-1)


def splitmix64_at(seed: int, i: int) -> int:
    """The i-th (0-based) output of the SplitMix64 stream seeded with ``seed``."""
    return int(_load().synth_splitmix64_at(seed & (2**64 - 1), i))


def i32_uniform(n: int, seed: int, out=None, nthreads=None) -> np.ndarray:
    a = _out(out, n, np.int32)
    _load().synth_i32_uniform(a.ctypes.data, n, seed, _threads(nthreads))
    return a


def i32_mod(n: int, seed: int, m: int, out=None, nthreads=None) -> np.ndarray:
    a = _out(out, n, np.int32)
    _load().synth_i32_mod(a.ctypes.data, n, seed, m, _threads(nthreads))
    return a


def i32_ascending(n: int, out=None, nthreads=None) -> np.ndarray:
    if n > 2**31:
        raise ValueError("ascending int32 input needs n <= 2^31")
    a = _out(out, n, np.int32)
    _load().synth_i32_ascending(a.ctypes.data, n, _threads(nthreads))
    return a


def f32_normal(n: int, seed: int, out=None, nthreads=None) -> np.ndarray:
    a = _out(out, n, np.float32)
    _load().synth_f32_normal(a.ctypes.data, n, seed, _threads(nthreads))
    return a


def f32_rows_tied(rows: int, cols: int, seed: int, frac: float = 0.01, out=None, nthreads=None) -> np.ndarray:
    """N(0,1) rows with floor(frac*cols) positions per row set to the row max."""
    a = _out(out, rows * cols, np.float32)
    f32_normal(rows * cols, seed, out=a, nthreads=nthreads)
    m = int(frac * cols)
    _load().synth_f32_force_ties(a.ctypes.data, rows, cols, m, seed, _threads(nthreads))
    return a.reshape(rows, cols)


def f32_rows_normal(rows: int, cols: int, seed: int, out=None, nthreads=None) -> np.ndarray:
    """The same N(0,1) rows without the tie forcing."""
    a = _out(out, rows * cols, np.float32)
    f32_normal(rows * cols, seed, out=a, nthreads=nthreads)
    return a.reshape(rows, cols)


# Named workloads: the int32 ones as (kind, n, seed) and the row one as
# (rows, cols, seed, tie fraction).  Sizes follow the TopK pages' benchmark
# table (1e7 / 1e8 / 1e9 elements, top 20) plus a small 2^20 case.
I32_WORKLOADS = {
    "i32_uniform_2p20": ("uniform", 1 << 20, 0),
    "i32_uniform_1e7": ("uniform", 10**7, 1),
    "i32_uniform_1e8": ("uniform", 10**8, 2),
    "i32_uniform_1e9": ("uniform", 10**9, 3),
    "i32_ascending_1e9": ("ascending", 10**9, None),
    "i32_dup1000_1e9": ("mod1000", 10**9, 4),
}

ROWS_WORKLOAD = {"rows": 4096, "cols": 32768, "seed": 5, "tie_frac": 0.01, "k": 64}


def i32_workload(name: str, out=None, nthreads=None) -> np.ndarray:
    kind, n, seed = I32_WORKLOADS[name]
    if kind == "uniform":
        return i32_uniform(n, seed, out=out, nthreads=nthreads)
    if kind == "ascending":
        return i32_ascending(n, out=out, nthreads=nthreads)
    if kind == "mod1000":
        return i32_mod(n, seed, 1000, out=out, nthreads=nthreads)
    raise KeyError(name)
