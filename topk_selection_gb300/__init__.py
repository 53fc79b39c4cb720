"""TopK selection on one GB300 (sm_103a): thin Python binding of libtopk.so.

Argument marshalling only -- every step of the selection runs in the CUDA
kernels behind the C ABI declared in include/topk.h.  PyTorch supplies device
memory and the current stream.  There is no CPU fallback: if the library has
not been built, importing the binding raises.

    topk_i32(x, k)          -> int32 tensor [k], the k largest values, descending
    topk_rows_f32(x, k)     -> (float32 [rows, k], int32 [rows, k]) per-row best
                               values and their columns; lower column wins ties

Both accept CUDA tensors (asynchronous on the current stream) or CPU tensors
(the library stages them through device memory and returns when done).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = ["topk_i32", "topk_rows_f32", "topk_i32_ptr", "topk_rows_f32_ptr", "TopKError", "MAX_K", "MAX_K_ROWS",
           "status_string", "release_workspace", "launch_count", "last_cuda_error", "library_path",
           "check_stream", "set_option", "OPT_STAGE2_CAP", "OPT_RADIX_CAP", "OPT_RADIX_SAMPLE_RANK",
           "reduce", "reduce_ptr", "REDUCE_OPS", "topk_items_f32", "topk_items_f32_ptr", "sort_u32",
           "sort_u32_ptr"]

MAX_K = 131072      # topk_i32, topk_u32, topk_f32
NOALLOC_MAX_K = 32768  # topk_i32_noalloc
MAX_K_ROWS = 1024   # topk_rows_f32
(TOPK_OK, TOPK_ERR_INVALID_ARG, TOPK_ERR_UNSUPPORTED, TOPK_ERR_NO_MEMORY, TOPK_ERR_CUDA,
 TOPK_ERR_DEVICE_TIMEOUT) = range(6)


class TopKError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def _load():
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    lib.topk_i32.argtypes = [vp, sz, ci, vp, vp]
    lib.topk_i32.restype = ci
    lib.topk_rows_f32.argtypes = [vp, ci, ci, ci, vp, vp, vp]
    lib.topk_rows_f32.restype = ci
    lib.topk_status_string.argtypes = [ci]
    lib.topk_status_string.restype = ctypes.c_char_p
    lib.topk_last_cuda_error.argtypes = []
    lib.topk_last_cuda_error.restype = ci
    lib.topk_release_workspace.argtypes = []
    lib.topk_release_workspace.restype = ci
    lib.topk_launch_count.argtypes = []
    lib.topk_launch_count.restype = ctypes.c_ulonglong
    lib.topk_check_stream.argtypes = [vp]
    lib.topk_check_stream.restype = ci
    lib.topk_set_option.argtypes = [ci, ci]
    lib.topk_set_option.restype = ci
    lib.topk_reduce_i32.argtypes = [vp, sz, ci, vp, vp]
    lib.topk_reduce_i32.restype = ci
    lib.topk_reduce_f32.argtypes = [vp, sz, ci, vp, vp]
    lib.topk_reduce_f32.restype = ci
    lib.topk_items_f32.argtypes = [vp, vp, vp, sz, ci, vp, vp, vp, vp]
    lib.topk_items_f32.restype = ci
    lib.topk_sort_u32.argtypes = [vp, vp, sz, vp, vp, vp]
    lib.topk_sort_u32.restype = ci
    lib.topk_u32.argtypes = [vp, sz, ci, vp, vp]
    lib.topk_u32.restype = ci
    lib.topk_f32.argtypes = [vp, sz, ci, vp, vp]
    lib.topk_f32.restype = ci
    lib.topk_last_launch_early.argtypes = []
    lib.topk_last_launch_early.restype = ci
    return lib


_lib = _load()


def status_string(status: int) -> str:
    return _lib.topk_status_string(int(status)).decode()


def last_cuda_error() -> int:
    return int(_lib.topk_last_cuda_error())


def release_workspace() -> None:
    rc = _lib.topk_release_workspace()
    if rc != TOPK_OK:
        raise TopKError(rc, "topk_release_workspace")


def launch_count() -> int:
    return int(_lib.topk_launch_count())


def last_launch_early() -> bool:
    """Whether this thread's last TopK launch may start while the previous
    kernel on its stream finishes (topk_last_launch_early)."""
    return bool(_lib.topk_last_launch_early())


OPT_STAGE2_CAP = 1
OPT_RADIX_CAP = 2
OPT_RADIX_SAMPLE_RANK = 3
OPT_STREAM_STATIC = 4
OPT_NO_EARLY_START = 5
OPT_FAULT_ALLOC = 6
OPT_SORT_SPINS = 7
OPT_SORT_WITHHOLD = 8


def set_option(option: int, value: int) -> None:
    """Process-wide option (see topk_set_option in include/topk.h)."""
    rc = _lib.topk_set_option(int(option), int(value))
    if rc != TOPK_OK:
        raise TopKError(rc, "topk_set_option")


def check_stream(stream=None, device=None) -> None:
    """Wait for the stream and raise TopKError if a kernel's bounded
    device-side wait gave up there (its results would not be valid)."""
    if device is None and torch.cuda.is_available():
        device = torch.cuda.current_device()
    rc = _lib.topk_check_stream(ctypes.c_void_p(_stream_handle(stream, device)))
    if rc != TOPK_OK:
        raise TopKError(rc, "topk_check_stream")


def _stream_handle(stream, device) -> int:
    if stream is None:
        if device is None:
            return 0
        stream = torch.cuda.current_stream(device)
    return int(getattr(stream, "cuda_stream", stream))


def topk_i32_ptr(in_ptr: int, n: int, k: int, out_ptr: int, stream: int = 0) -> int:
    """Raw C-ABI call; returns the status code."""
    return int(_lib.topk_i32(ctypes.c_void_p(in_ptr), n, k, ctypes.c_void_p(out_ptr), ctypes.c_void_p(stream)))


def topk_rows_f32_ptr(in_ptr: int, rows: int, cols: int, k: int, vals_ptr: int, idx_ptr: int,
                      stream: int = 0) -> int:
    """Raw C-ABI call; returns the status code."""
    return int(_lib.topk_rows_f32(ctypes.c_void_p(in_ptr), rows, cols, k, ctypes.c_void_p(vals_ptr),
                                  ctypes.c_void_p(idx_ptr), ctypes.c_void_p(stream)))


def _check_input(x: torch.Tensor, dtype, name):
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def topk_i32(x: torch.Tensor, k: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The k largest values of int32 tensor x (flattened), sorted descending."""
    _check_input(x, torch.int32, "x")
    if out is None:
        out = torch.empty(max(int(k), 0), dtype=torch.int32, device=x.device)
    _check_input(out, torch.int32, "out")
    if out.numel() != k:
        raise ValueError("out must have k elements")
    dev = x.device if x.is_cuda else (out.device if out.is_cuda else None)
    with torch.cuda.device(dev) if dev is not None else _null():
        rc = topk_i32_ptr(x.data_ptr(), x.numel(), int(k), out.data_ptr(), _stream_handle(stream, dev))
    if rc != TOPK_OK:
        raise TopKError(rc, "topk_i32")
    return out


def topk_u32_ptr(in_ptr: int, n: int, k: int, out_ptr: int, stream: int = 0) -> int:
    """Raw C-ABI call; returns the status code."""
    return int(_lib.topk_u32(ctypes.c_void_p(in_ptr), n, k, ctypes.c_void_p(out_ptr), ctypes.c_void_p(stream)))


def topk_f32_ptr(in_ptr: int, n: int, k: int, out_ptr: int, stream: int = 0) -> int:
    """Raw C-ABI call; returns the status code."""
    return int(_lib.topk_f32(ctypes.c_void_p(in_ptr), n, k, ctypes.c_void_p(out_ptr), ctypes.c_void_p(stream)))


def _topk_words(fn, name, x, k, out, stream, dtypes):
    if x.dtype not in dtypes:
        raise TypeError(f"x must be one of {dtypes}, got {x.dtype}")
    _check_input(x, x.dtype, "x")
    if out is None:
        out = torch.empty(max(int(k), 0), dtype=x.dtype, device=x.device)
    _check_input(out, x.dtype, "out")
    if out.numel() != k:
        raise ValueError("out must have k elements")
    dev = x.device if x.is_cuda else (out.device if out.is_cuda else None)
    with torch.cuda.device(dev) if dev is not None else _null():
        rc = fn(x.data_ptr(), x.numel(), int(k), out.data_ptr(), _stream_handle(stream, dev))
    if rc != TOPK_OK:
        raise TopKError(rc, name)
    return out


def topk_u32(x: torch.Tensor, k: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The k largest of the uint32 keys in x (flattened), descending.  x may
    be torch.uint32, or int32 holding the keys' bits (out has x's dtype)."""
    return _topk_words(topk_u32_ptr, "topk_u32", x, k, out, stream, (torch.uint32, torch.int32))


def topk_f32(x: torch.Tensor, k: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The k largest float32 values of x (flattened) under IEEE 754 totalOrder,
    descending (see topk_f32 in include/topk.h)."""
    return _topk_words(topk_f32_ptr, "topk_f32", x, k, out, stream, (torch.float32,))


def topk_rows_f32(x: torch.Tensor, k: int, vals: torch.Tensor | None = None, idx: torch.Tensor | None = None,
                  stream=None):
    """Per-row TopK of a 2-D float32 tensor: (values [rows, k], columns [rows, k])."""
    _check_input(x, torch.float32, "x")
    if x.dim() != 2:
        raise ValueError("x must be 2-D (rows, cols)")
    rows, cols = x.shape
    if vals is None:
        vals = torch.empty((rows, max(int(k), 0)), dtype=torch.float32, device=x.device)
    if idx is None:
        idx = torch.empty((rows, max(int(k), 0)), dtype=torch.int32, device=x.device)
    _check_input(vals, torch.float32, "vals")
    _check_input(idx, torch.int32, "idx")
    if vals.numel() != rows * k or idx.numel() != rows * k:
        raise ValueError("vals and idx must have rows*k elements")
    dev = x.device if x.is_cuda else None
    with torch.cuda.device(dev) if dev is not None else _null():
        rc = topk_rows_f32_ptr(x.data_ptr(), rows, cols, int(k), vals.data_ptr(), idx.data_ptr(),
                               _stream_handle(stream, dev))
    if rc != TOPK_OK:
        raise TopKError(rc, "topk_rows_f32")
    return vals, idx


def topk_items_f32_ptr(score_ptr: int, item_ptr: int, keep_ptr: int, n: int, k: int, out_score_ptr: int,
                       out_item_ptr: int, out_count_ptr: int, stream: int = 0) -> int:
    """Raw C-ABI call (0 for a null item, keep or out_count); returns the status code."""
    vp = ctypes.c_void_p
    return int(_lib.topk_items_f32(vp(score_ptr), vp(item_ptr or None), vp(keep_ptr or None), n, k,
                                   vp(out_score_ptr), vp(out_item_ptr), vp(out_count_ptr or None), vp(stream)))


def topk_items_f32(score: torch.Tensor, k: int, item: torch.Tensor | None = None, keep: torch.Tensor | None = None,
                   stream=None):
    """Score-keyed TopK with item ids over CUDA tensors: (scores [k] float32,
    items [k] int64, count) -- see topk_items_f32 in include/topk.h."""
    _check_input(score, torch.float32, "score")
    if not score.is_cuda:
        raise ValueError("score must be a CUDA tensor")
    n = score.numel()
    if item is not None:
        _check_input(item, torch.int64, "item")
        if item.numel() != n:
            raise ValueError("item must match score")
    if keep is not None:
        if keep.dtype == torch.bool:
            keep = keep.view(torch.uint8)
        _check_input(keep, torch.uint8, "keep")
        if keep.numel() != n:
            raise ValueError("keep must match score")
    dev = score.device
    out_score = torch.empty(max(int(k), 0), dtype=torch.float32, device=dev)
    out_item = torch.empty(max(int(k), 0), dtype=torch.int64, device=dev)
    out_count = torch.empty(1, dtype=torch.int64, device=dev)
    with torch.cuda.device(dev):
        rc = topk_items_f32_ptr(score.data_ptr(), item.data_ptr() if item is not None else 0,
                                keep.data_ptr() if keep is not None else 0, n, int(k), out_score.data_ptr(),
                                out_item.data_ptr(), out_count.data_ptr(), _stream_handle(stream, dev))
    if rc != TOPK_OK:
        raise TopKError(rc, "topk_items_f32")
    return out_score, out_item, out_count


def sort_u32_ptr(keys_ptr: int, vals_ptr: int, n: int, keys_out_ptr: int, vals_out_ptr: int, stream: int = 0) -> int:
    """Raw C-ABI call (0 for null value pointers); returns the status code."""
    vp = ctypes.c_void_p
    return int(_lib.topk_sort_u32(vp(keys_ptr), vp(vals_ptr or None), n, vp(keys_out_ptr), vp(vals_out_ptr or None),
                                  vp(stream)))


def sort_u32(keys: torch.Tensor, vals: torch.Tensor | None = None, stream=None):
    """Stable ascending radix sort of uint32 keys (a CUDA tensor of dtype
    torch.uint32, or int32 reinterpreted as uint32), carrying uint32 values:
    (sorted keys, sorted values or None)."""
    def as_u32(t, name):
        if t.dtype == torch.int32:
            return t
        if t.dtype == getattr(torch, "uint32", None):
            return t
        raise TypeError(f"{name} must be uint32 (or int32 holding uint32 bits)")
    keys = as_u32(keys, "keys")
    if not keys.is_cuda or not keys.is_contiguous():
        raise ValueError("keys must be a contiguous CUDA tensor")
    if vals is not None:
        vals = as_u32(vals, "vals")
        if not vals.is_cuda or not vals.is_contiguous() or vals.numel() != keys.numel():
            raise ValueError("vals must be a contiguous CUDA tensor matching keys")
    ko = torch.empty_like(keys)
    vo = torch.empty_like(vals) if vals is not None else None
    dev = keys.device
    with torch.cuda.device(dev):
        rc = sort_u32_ptr(keys.data_ptr(), vals.data_ptr() if vals is not None else 0, keys.numel(), ko.data_ptr(),
                          vo.data_ptr() if vo is not None else 0, _stream_handle(stream, dev))
    if rc != TOPK_OK:
        raise TopKError(rc, "topk_sort_u32")
    return ko, vo


REDUCE_OPS = {"sum": 0, "max": 1, "min": 2}


def reduce_ptr(in_ptr: int, n: int, is_float: bool, op: int, out_ptr: int, stream: int = 0) -> int:
    """Raw C-ABI call (topk_reduce_f32 if is_float else topk_reduce_i32); returns the status code."""
    fn = _lib.topk_reduce_f32 if is_float else _lib.topk_reduce_i32
    return int(fn(ctypes.c_void_p(in_ptr), n, op, ctypes.c_void_p(out_ptr), ctypes.c_void_p(stream)))


def reduce(x: torch.Tensor, op: str, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Sum, max or min of an int32 or float32 tensor (flattened).  Returns a
    one-element tensor: int64 for int32 input (exact sum), float64 for
    float32 input (see topk_reduce_f32 in include/topk.h for its rules)."""
    if x.dtype not in (torch.int32, torch.float32):
        raise TypeError("x must be int32 or float32")
    _check_input(x, x.dtype, "x")
    is_float = x.dtype == torch.float32
    odt = torch.float64 if is_float else torch.int64
    if out is None:
        out = torch.empty(1, dtype=odt, device=x.device)
    _check_input(out, odt, "out")
    if out.numel() != 1:
        raise ValueError("out must have one element")
    dev = x.device if x.is_cuda else (out.device if out.is_cuda else None)
    with torch.cuda.device(dev) if dev is not None else _null():
        rc = reduce_ptr(x.data_ptr(), x.numel(), is_float, REDUCE_OPS[op], out.data_ptr(), _stream_handle(stream, dev))
    if rc != TOPK_OK:
        raise TopKError(rc, "topk_reduce_f32" if is_float else "topk_reduce_i32")
    return out


class _null:
    def __enter__(self):
        return None

    def __exit__(self, *a):
        return False
