"""Radix sort (uint32 keys, optional uint32 values) on the GPU, through the
C ABI, against the oracle: keys and values must be identical (a stable
sort, so values of equal keys keep their input order)."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tk():
    import topk_selection_gb300

    yield topk_selection_gb300
    topk_selection_gb300.check_stream()


def gpu_sort(tk, keys, vals=None):
    dk = torch.from_numpy(keys.view(np.int32)).cuda()
    dv = None if vals is None else torch.from_numpy(vals.view(np.int32)).cuda()
    ko, vo = tk.sort_u32(dk, dv)
    torch.cuda.synchronize()
    return ko.cpu().numpy().view(np.uint32), None if vo is None else vo.cpu().numpy().view(np.uint32)


def check(tk, keys, with_vals=True):
    vals = np.arange(keys.size, dtype=np.uint32) * np.uint32(2654435761) if with_vals else None
    gk, gv = gpu_sort(tk, keys, vals)
    ek, ev = oracle.sort_u32(keys, vals)
    assert np.array_equal(gk, ek), (keys.size, np.nonzero(gk != ek)[0][:5])
    if with_vals:
        assert np.array_equal(gv, ev), (keys.size, np.nonzero(gv != ev)[0][:5])


def make(kind, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "uniform":
        return synth.i32_uniform(n, seed).view(np.uint32).copy()
    if kind == "few":
        return rng.integers(0, 5, size=n, dtype=np.uint64).astype(np.uint32) * np.uint32(0x01010101)
    if kind == "equal":
        return np.full(n, 0xDEADBEEF, dtype=np.uint32)
    if kind == "descending":
        return (np.uint64(0xFFFFFFFF) - np.arange(n, dtype=np.uint64)).astype(np.uint32)
    if kind == "sorted":
        return np.sort(rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32))
    if kind == "extremes":
        return rng.choice(np.array([0, 0xFFFFFFFF, 0x80000000, 0x7FFFFFFF], dtype=np.uint32), size=n)
    if kind == "high_byte":
        return (rng.integers(0, 256, size=n, dtype=np.uint64) << np.uint64(24)).astype(np.uint32)
    raise KeyError(kind)


SIZES = [1, 2, 3, 31, 32, 33, 4095, 4096, 4097, 8191, 8192, 8193, 16385, 65537, 1_000_003]  # around one and two tiles


@pytest.mark.parametrize("kind", ["uniform", "few", "equal", "descending", "sorted", "extremes", "high_byte"])
def test_sizes(tk, kind):
    for n in SIZES:
        x = make(kind, n, n)
        check(tk, x, with_vals=True)
        check(tk, x, with_vals=False)


def test_back_to_back_different_sizes(tk):
    # Tile counters and look-back words are reused call after call.
    for n in (5000, 1_000_001, 4096, 123_457, 1_000_001, 7):
        check(tk, make("uniform", n, n + 1))
        check(tk, make("few", n, n + 2), with_vals=False)


def test_large(tk):
    x = make("uniform", 16_777_219, 41)
    check(tk, x, with_vals=True)
    y = make("few", 16_777_219, 42)
    check(tk, y, with_vals=True)
