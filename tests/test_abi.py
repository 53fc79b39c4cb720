"""The C ABI without a GPU: the library loads, exports every function that
include/*.h declares, and rejects bad arguments on the host before any CUDA
call (so these run on a machine without a GPU)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import topk_selection_gb300 as tk

    return tk._lib


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(topk_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("topk_i32", "topk_rows_f32", "topk_status_string", "topk_release_workspace",
                     "topk_last_cuda_error", "topk_launch_count"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libtopk.so does not export {name}"


def test_status_strings(lib):
    import topk_selection_gb300 as tk

    assert tk.status_string(0) == "ok"
    assert tk.status_string(1) == "invalid argument"
    assert tk.status_string(2) == "unsupported size"
    assert tk.status_string(5) == "a device-side wait gave up"
    assert tk.status_string(99) == "unknown status"


# Fake, never-dereferenced addresses: the argument checks return before any
# pointer is used or any CUDA call is made.
A, B, C = 0x10000000, 0x20000000, 0x30000000


@pytest.mark.parametrize("args,status", [
    ((0, 100, 5, B), 1),          # null input
    ((A, 100, 5, 0), 1),          # null output
    ((A, 0, 1, B), 1),            # n == 0
    ((A, 100, 0, B), 1),          # k < 1
    ((A, 100, -3, B), 1),         # k < 1
    ((A, 100, 101, B), 1),        # k > n
    ((A + 2, 100, 5, B), 1),      # misaligned input
    ((A, 100, 5, B + 1), 1),      # misaligned output
    ((A, 100, 5, A + 40), 1),     # output overlaps input
    ((A, 200000, 131073, B), 2),  # k above the maximum
    ((B, (1 << 40) + 4, 5, A), 2),  # n above the maximum
])
def test_topk_i32_argument_errors(lib, args, status):
    import topk_selection_gb300 as tk

    assert tk.topk_i32_ptr(*args) == status


@pytest.mark.parametrize("args,status", [
    ((0, 4, 8, 2, B, C), 1),        # null input
    ((A, 4, 8, 2, 0, C), 1),        # null vals
    ((A, 4, 8, 2, B, 0), 1),        # null idx
    ((A, 0, 8, 2, B, C), 1),        # rows < 1
    ((A, 4, 0, 1, B, C), 1),        # cols < 1
    ((A, 4, 8, 0, B, C), 1),        # k < 1
    ((A, 4, 8, 9, B, C), 1),        # k > cols
    ((A, 4, 8, 2, B, B + 8), 1),    # vals and idx overlap
    ((A, 4, 8, 2, A + 4, C), 1),    # vals overlaps the input
    ((A, 4, 2048, 1025, B, C), 2),  # k above the row maximum
])
def test_topk_rows_argument_errors(lib, args, status):
    import topk_selection_gb300 as tk

    assert tk.topk_rows_f32_ptr(*args) == status


def test_python_binding_rejects_wrong_types(lib):
    import torch

    import topk_selection_gb300 as tk

    with pytest.raises(TypeError):
        tk.topk_i32(torch.zeros(10, dtype=torch.int64), 3)
    with pytest.raises(TypeError):
        tk.topk_rows_f32(torch.zeros(2, 10, dtype=torch.float64), 3)
    with pytest.raises(ValueError):
        tk.topk_rows_f32(torch.zeros(10, dtype=torch.float32), 3)
    with pytest.raises(ValueError):
        tk.topk_i32(torch.zeros(20, dtype=torch.int32)[::2], 3)
    with pytest.raises(tk.TopKError) as e:
        tk.topk_i32(torch.zeros(10, dtype=torch.int32), 11)
    assert e.value.status == 1


def test_reduce_and_items_argument_errors(lib):
    import topk_selection_gb300 as tk

    buf = (ctypes.c_int32 * 64)()
    out = (ctypes.c_int64 * 64)()
    p, o = ctypes.addressof(buf), ctypes.addressof(out)
    f = lib.topk_reduce_i32
    assert f(None, 10, 0, o, None) == 1              # null input
    assert f(p, 10, 0, None, None) == 1              # null output
    assert f(p, 0, 0, o, None) == 1                  # n == 0
    assert f(p, 10, 3, o, None) == 1                 # unknown op
    assert f(p, 10, -1, o, None) == 1
    assert f(p + 1, 10, 0, o, None) == 1             # misaligned input
    assert f(p, 10, 0, o + 4, None) == 1             # misaligned output
    assert lib.topk_reduce_f32(p, 10, 1, p + 8, None) == 1  # output overlaps input
    g = lib.topk_items_f32
    assert g(None, None, None, 10, 1, p, o, None, None) == 1   # null score
    assert g(p, None, None, 10, 1, None, o, None, None) == 1   # null out_score
    assert g(p, None, None, 0, 1, p + 128, o, None, None) == 1  # n == 0
    assert g(p, None, None, 10, 11, p + 128, o, None, None) == 1  # k > n
    assert g(p, None, None, 10, 0, p + 128, o, None, None) == 1   # k < 1
    assert g(p, None, None, 10, 2, p, o, None, None) == 1      # out_score overlaps score
    assert g(p, o + 4, None, 10, 2, p + 128, o + 64, None, None) == 1  # misaligned item
    h = lib.topk_sort_u32
    assert h(None, None, 10, p, None, None) == 1            # null keys
    assert h(p, None, 0, p + 128, None, None) == 1          # n == 0
    assert h(p, p + 64, 10, p + 128, None, None) == 1       # values without an output for them
    assert h(p, None, 10, p + 16, None, None) == 1          # output overlaps input
    assert h(p + 2, None, 10, p + 128, None, None) == 1     # misaligned
    assert tk.OPT_STAGE2_CAP == 1


def test_launch_counter_starts_at_zero_without_gpu(lib):
    import topk_selection_gb300 as tk

    assert tk.launch_count() >= 0


def test_set_option_validation(lib):
    import topk_selection_gb300 as tk

    for bad in (-1, 1, 3, 100):
        assert tk._lib.topk_set_option(tk.OPT_STAGE2_CAP, bad) == 1
    assert tk._lib.topk_set_option(99, 0) == 1
    assert tk._lib.topk_set_option(tk.OPT_STAGE2_CAP, 64) == 0
    assert tk._lib.topk_set_option(tk.OPT_STAGE2_CAP, 0) == 0
    for opt in (tk.OPT_RADIX_CAP, tk.OPT_RADIX_SAMPLE_RANK):
        assert tk._lib.topk_set_option(opt, -1) == 1
        assert tk._lib.topk_set_option(opt, 5) == 0
        assert tk._lib.topk_set_option(opt, 0) == 0
    text = open(os.path.join(ROOT, "include", "topk.h")).read()
    for name, value in (("TOPK_OPT_STAGE2_CAP", tk.OPT_STAGE2_CAP), ("TOPK_OPT_RADIX_CAP", tk.OPT_RADIX_CAP),
                        ("TOPK_OPT_RADIX_SAMPLE_RANK", tk.OPT_RADIX_SAMPLE_RANK)):
        assert re.search(r"%s = %d\b" % (name, value), text), name


def test_header_limits_match_binding(lib):
    import topk_selection_gb300 as tk

    text = open(os.path.join(ROOT, "include", "topk.h")).read()
    assert re.search(r"#define TOPK_MAX_K\s+%d\b" % tk.MAX_K, text)
    assert re.search(r"#define TOPK_MAX_K_ROWS\s+%d\b" % tk.MAX_K_ROWS, text)


def test_options_accept_and_reject(lib):
    import topk_selection_gb300 as tk

    for opt, good, bad in ((tk.OPT_NO_EARLY_START, (1, 0), (2, -1)), (tk.OPT_FAULT_ALLOC, (1, 0), (2, -1)),
                           (tk.OPT_SORT_SPINS, (1, 0), (-1,)), (tk.OPT_SORT_WITHHOLD, (1, 0), (-1, 2)), (tk.OPT_STREAM_STATIC, (1, 101, 0), (102, -1)),
                           (tk.OPT_STAGE2_CAP, (64, 0), (3, 1))):
        for v in good:
            tk.set_option(opt, v)
        for v in bad:
            with pytest.raises(tk.TopKError):
                tk.set_option(opt, v)
    with pytest.raises(tk.TopKError):
        tk.set_option(99, 0)


@pytest.mark.parametrize("fn", ["topk_u32_ptr", "topk_f32_ptr"])
def test_u32_f32_argument_errors(lib, fn):
    import topk_selection_gb300 as tk

    f = getattr(tk, fn)
    assert f(0, 100, 5, B) == 1
    assert f(A, 0, 1, B) == 1
    assert f(A, 100, 101, B) == 1
    assert f(A + 2, 100, 5, B) == 1
    assert f(A, 100, 5, A + 40) == 1
    assert f(A, 200000, 131073, B) == 2
