"""topk_i32_noalloc: the int32 TopK whose scratch is a fixed device array.

It serves callers that cannot allocate device memory: a plugin enqueue hook
that must not allocate, a process whose memory another allocator's pool has
already claimed, a loop that cannot take cudaMalloc's implicit
synchronisation.  Its results must equal the oracle's and topk_i32's
exactly (int32 output, bit-exact as in every other int32 test), call after
call, since every call reuses the same array.

This file is collected last on purpose, so a run that stops at its first
failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def entry():
    import topk_selection_gb300 as tk

    f = tk._lib.topk_i32_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return tk, f


def run_noalloc(f, x, k, stream, out=None):
    if out is None:
        out = torch.empty(k, dtype=torch.int32, device=x.device)
    rc = f(x.data_ptr(), x.numel(), k, out.data_ptr(), stream.cuda_stream)
    assert rc == 0, rc
    return out


def test_noalloc_matches_oracle_and_topk_i32_on_two_calls_in_a_row(entry):
    tk, f = entry
    stream = torch.cuda.current_stream()
    # Two different inputs back to back: a call that leaves a high threshold
    # behind, then one whose answer lies far below it.
    a = synth.i32_uniform(3_000_017, 41)
    b = synth.i32_mod(2_500_003, 42, 1000) - np.int32(5000)
    for x, k in ((a, 20), (b, 100)):
        d = torch.from_numpy(x).cuda()
        got = run_noalloc(f, d, k, stream)
        cached = tk.topk_i32(d, k)
        torch.cuda.synchronize()
        exp = oracle.topk_i32(x, k)
        assert np.array_equal(got.cpu().numpy(), exp), (k, got[:5], exp[:5])
        assert np.array_equal(cached.cpu().numpy(), exp), k


def test_noalloc_large_k_and_small_input(entry):
    tk, f = entry
    stream = torch.cuda.current_stream()
    for n, k in ((5, 3), (100_003, 1024), (4_194_311, 1000), (3_000_017, 32768)):
        x = synth.i32_uniform(n, n)
        d = torch.from_numpy(x).cuda()
        exp = oracle.topk_i32(x, k)
        for _ in range(2):
            got = run_noalloc(f, d, k, stream)
            cached = tk.topk_i32(d, k)
            torch.cuda.synchronize()
            assert np.array_equal(got.cpu().numpy(), exp), (n, k)
            assert np.array_equal(cached.cpu().numpy(), exp), (n, k)


def test_noalloc_and_cached_calls_chained_on_one_stream(entry):
    # Calls of both entry points feed each other on one stream: every call
    # must see the previous one's output finished, whichever entry point
    # launched it.
    tk, f = entry
    x = synth.i32_uniform(3_000_029, 43)
    d = torch.from_numpy(x).cuda()
    s = torch.cuda.Stream()
    exp = oracle.topk_i32(x, 3000)
    with torch.cuda.stream(s):
        for _ in range(3):
            a = run_noalloc(f, d, 3000, s)          # large-k plan, fixed scratch
            b = tk.topk_i32(a, 100, stream=s)       # cached workspace, streaming, reads a
            assert not tk.last_launch_early()       # its predecessor is a no-alloc launch
            c = run_noalloc(f, b, 50, s)            # fixed scratch, streaming, reads b
            e = tk.topk_i32(c, 20, stream=s)        # reads c
            assert not tk.last_launch_early()
            g = tk.topk_i32(d, 128, stream=s)       # independent input
            h = run_noalloc(f, g, 1, s)             # reads g
    s.synchronize()
    assert np.array_equal(a.cpu().numpy(), exp)
    assert np.array_equal(b.cpu().numpy(), exp[:100])
    assert np.array_equal(c.cpu().numpy(), exp[:50])
    assert np.array_equal(e.cpu().numpy(), exp[:20])
    assert np.array_equal(g.cpu().numpy(), exp[:128])
    assert h.cpu().numpy()[0] == exp[0]


def test_noalloc_allocates_no_device_memory(entry):
    tk, f = entry
    stream = torch.cuda.current_stream()
    x = torch.from_numpy(synth.i32_uniform(2_000_003, 44)).cuda()
    outs = {k: torch.empty(k, dtype=torch.int32, device="cuda") for k in (20, 100, 1000)}
    for k, o in outs.items():  # warm-up: loads the kernels' code and the array's address
        run_noalloc(f, x, k, stream, o)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(10):
        for k, o in outs.items():
            run_noalloc(f, x, k, stream, o)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)


def test_noalloc_rejects_what_it_cannot_take(entry):
    tk, f = entry
    x2 = torch.zeros(40000, dtype=torch.int32, device="cuda")
    out = torch.empty(32769, dtype=torch.int32, device="cuda")
    assert f(x2.data_ptr(), 40000, 32769, out.data_ptr(), None) == 2  # k above the maximum
    xh = torch.zeros(5000, dtype=torch.int32)
    assert f(xh.data_ptr(), 5000, 20, out.data_ptr(), None) == 1   # host input: would need staging
    assert f(x2.data_ptr() + 1, 1000, 20, out.data_ptr(), None) == 1  # misaligned input
    assert f(x2.data_ptr(), 40000, 20, x2.data_ptr() + 400, None) == 1  # output inside the input
    assert f(x2.data_ptr(), 0, 1, out.data_ptr(), None) == 1  # empty input
    assert f(x2.data_ptr(), 10, 11, out.data_ptr(), None) == 1  # k above n
