"""topk_i32_noalloc: the int32 TopK whose scratch is a fixed device array.

It serves callers that cannot allocate device memory (a plugin enqueue hook
that must not allocate, a process whose memory another allocator's pool has
already claimed, a loop that cannot take cudaMalloc's implicit
synchronisation).  Its results must equal topk_i32's exactly (int32 output,
bit-exact as in every other int32 test), call after call, since every call
reuses the same array.

This file is collected last on purpose, so a run that stops at its first
failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def entry():
    import topk_selection_gb300 as tk

    f = tk._lib.topk_i32_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return tk, f


def run_noalloc(f, x, k, stream):
    out = torch.empty(k, dtype=torch.int32, device=x.device)
    rc = f(x.data_ptr(), x.numel(), k, out.data_ptr(), stream.cuda_stream)
    assert rc == 0, rc
    return out


def test_noalloc_matches_topk_i32_on_two_calls_in_a_row(entry):
    tk, f = entry
    stream = torch.cuda.current_stream()
    # Two different inputs back to back: a call that leaves a high threshold
    # behind, then one whose answer lies far below it.
    a = torch.from_numpy(synth.i32_uniform(3_000_017, 41)).cuda()
    b = torch.from_numpy(synth.i32_mod(2_500_003, 42, 1000) - np.int32(5000)).cuda()
    for x, k in ((a, 20), (b, 100)):
        got = run_noalloc(f, x, k, stream)
        exp = tk.topk_i32(x, k)
        torch.cuda.synchronize()
        assert torch.equal(got.cpu(), exp.cpu()), (k, got[:5], exp[:5])


def test_noalloc_large_k_and_small_input(entry):
    tk, f = entry
    stream = torch.cuda.current_stream()
    for n, k in ((5, 3), (100_003, 1024), (4_194_311, 1000), (3_000_017, 32768)):
        x = torch.from_numpy(synth.i32_uniform(n, n)).cuda()
        for _ in range(2):
            got = run_noalloc(f, x, k, stream)
            exp = tk.topk_i32(x, k)
            torch.cuda.synchronize()
            assert torch.equal(got.cpu(), exp.cpu()), (n, k)



def test_noalloc_and_cached_calls_chained_on_one_stream(entry):
    # Calls of both entry points feed each other on one stream: every call
    # must see the previous one's output finished, whichever entry point
    # launched it.
    tk, f = entry
    import oracle
    x = synth.i32_uniform(3_000_029, 43)
    d = torch.from_numpy(x).cuda()
    s = torch.cuda.Stream()
    exp = oracle.topk_i32(x, 3000)
    with torch.cuda.stream(s):
        for _ in range(3):
            a = run_noalloc(f, d, 3000, s)          # large-k plan, fixed scratch
            b = tk.topk_i32(a, 100, stream=s)       # cached workspace, streaming, reads a
            c = run_noalloc(f, b, 50, s)            # fixed scratch, streaming, reads b
            e = tk.topk_i32(c, 20, stream=s)        # reads c
            g = tk.topk_i32(d, 128, stream=s)       # independent input
            h = run_noalloc(f, g, 1, s)             # reads g
    s.synchronize()
    assert np.array_equal(a.cpu().numpy(), exp)
    assert np.array_equal(b.cpu().numpy(), exp[:100])
    assert np.array_equal(c.cpu().numpy(), exp[:50])
    assert np.array_equal(e.cpu().numpy(), exp[:20])
    assert np.array_equal(g.cpu().numpy(), exp[:128])
    assert h.cpu().numpy()[0] == exp[0]


def test_noalloc_rejects_what_it_cannot_take(entry):
    tk, f = entry
    x = torch.zeros(5000, dtype=torch.int32, device="cuda")
    x2 = torch.zeros(40000, dtype=torch.int32, device="cuda")
    out = torch.empty(32769, dtype=torch.int32, device="cuda")
    assert f(x2.data_ptr(), 40000, 32769, out.data_ptr(), None) == 2  # k above the maximum
    xh = torch.zeros(5000, dtype=torch.int32)
    assert f(xh.data_ptr(), 5000, 20, out.data_ptr(), None) == 1   # host input: would need staging
