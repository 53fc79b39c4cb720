"""Sum / max / min reductions on the GPU, through the C ABI, against the oracle.

int32 results and float32 max/min are compared exactly (value and sign of
zero; NaN as NaN).  The float32 sum is compared within the bound the two
arithmetics give: the GPU's float32 vector sums (pairwise, error <= 2u
of their magnitudes, u = 2^-24) added with compensation (error <= 2u more)
are within 4u = 2^-22 of sum|x| of the exact sum, plus the rounding of
folding them in double; the oracle's left-to-right double sum is within
n * 2^-53 * sum|x| of it.  The test allows (2^-22 + 2 n 2^-52) sum|x|.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

INT_MIN, INT_MAX = -(2**31), 2**31 - 1
OPS = ("sum", "max", "min")


@pytest.fixture(scope="module")
def tk():
    import topk_selection_gb300

    yield topk_selection_gb300
    topk_selection_gb300.check_stream()


def gpu_reduce(tk, x_np, op, offset=0):
    dt = torch.int32 if x_np.dtype == np.int32 else torch.float32
    buf = torch.empty(x_np.size + offset, dtype=dt, device="cuda")
    view = buf[offset:]
    view.copy_(torch.from_numpy(x_np))
    out = tk.reduce(view, op)
    torch.cuda.synchronize()
    return out.item()


def same(a, b):
    return (math.isnan(a) and math.isnan(b)) or (a == b and math.copysign(1.0, a) == math.copysign(1.0, b))


def f32_sum_ok(got, x, exp):
    if not math.isfinite(exp) or not math.isfinite(got):
        return same(got, exp)
    tol = (2.0 ** -22 + 2 * x.size * 2.0 ** -52) * float(np.abs(x.astype(np.float64)).sum())
    return abs(got - exp) <= tol


def check(tk, x, op, offset=0):
    got = gpu_reduce(tk, x, op, offset)
    if x.dtype == np.int32:
        exp = oracle.reduce_i32(x, op)
        assert got == exp, (op, x.size, got, exp)
    else:
        exp = oracle.reduce_f32(x, op)
        ok = f32_sum_ok(got, x, exp) if op == "sum" else same(got, exp)
        assert ok, (op, x.size, got, exp)


SIZES = [1, 2, 3, 4, 5, 7, 31, 33, 1023, 1025, 4097, 65537, 300_007, 2_000_003]


def make_i32(kind, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "uniform":
        return synth.i32_uniform(n, seed)
    if kind == "int_max":
        return np.full(n, INT_MAX, dtype=np.int32)
    if kind == "int_min":
        return np.full(n, INT_MIN, dtype=np.int32)
    if kind == "negative":
        return rng.integers(INT_MIN, 0, size=n, dtype=np.int64).astype(np.int32)
    if kind == "small":
        return rng.integers(-3, 4, size=n).astype(np.int32)
    raise KeyError(kind)


def make_f32(kind, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return synth.f32_normal(n, seed)
    if kind == "specials":
        pool = np.array([math.nan, math.inf, -math.inf, -0.0, 0.0, 1.0, -1.0, 3e38, -3e38, 1e-45],
                        dtype=np.float32)
        return pool[rng.integers(0, pool.size, n)]
    if kind == "zeros":
        return np.where(rng.random(n) < 0.5, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
    if kind == "neg_zeros":
        return np.full(n, -0.0, dtype=np.float32)
    if kind == "wide":
        return (rng.standard_normal(n) * np.exp2(rng.integers(-60, 60, n))).astype(np.float32)
    if kind == "one_inf":
        x = rng.standard_normal(n).astype(np.float32)
        x[n // 2] = math.inf
        return x
    if kind == "one_nan":
        x = rng.standard_normal(n).astype(np.float32)
        x[n - 1] = math.nan
        return x
    raise KeyError(kind)


@pytest.mark.parametrize("kind", ["uniform", "int_max", "int_min", "negative", "small"])
def test_i32_sizes(tk, kind):
    for n in SIZES:
        x = make_i32(kind, n, n)
        for op in OPS:
            check(tk, x, op)


@pytest.mark.parametrize("kind", ["normal", "specials", "zeros", "neg_zeros", "wide", "one_inf", "one_nan"])
def test_f32_sizes(tk, kind):
    for n in SIZES:
        x = make_f32(kind, n, n)
        for op in OPS:
            check(tk, x, op)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned(tk, offset):
    for n in (5, 6, 7, 1029, 262_147):
        check(tk, make_i32("uniform", n, offset), "sum", offset)
        check(tk, make_i32("negative", n, offset), "max", offset)
        check(tk, make_f32("normal", n, offset), "sum", offset)
        check(tk, make_f32("specials", n, offset), "min", offset)


def test_back_to_back_and_host_buffers(tk):
    x = make_i32("uniform", 1_000_003, 3)
    f = make_f32("normal", 1_000_003, 4)
    for _ in range(3):
        for op in OPS:
            check(tk, x, op)
            check(tk, f, op)
    # host tensors: the library stages them
    got = tk.reduce(torch.from_numpy(x), "sum").item()
    assert got == oracle.reduce_i32(x, "sum")
    got = tk.reduce(torch.from_numpy(f), "max").item()
    assert same(got, oracle.reduce_f32(f, "max"))


def test_reduce_and_topk_share_a_stream(tk):
    # The reduction's ticket lives in the same workspace as the TopK plans.
    x = make_i32("uniform", 2_000_003, 9)
    d = torch.from_numpy(x).cuda()
    for k in (20, 1000, 1):
        t = tk.topk_i32(d, k)
        s = tk.reduce(d, "sum")
        torch.cuda.synchronize()
        assert np.array_equal(t.cpu().numpy(), oracle.topk_i32(x, k))
        assert s.item() == oracle.reduce_i32(x, "sum")


def test_workload_1e8(tk):
    x = synth.i32_workload("i32_uniform_1e8")
    d = torch.from_numpy(x).cuda()
    for op in OPS:
        assert tk.reduce(d, op).item() == oracle.reduce_i32(x, op), op
    del d
    f = (x.astype(np.float64) * 2.0 ** -31).astype(np.float32)
    df = torch.from_numpy(f).cuda()
    got = tk.reduce(df, "sum").item()
    assert f32_sum_ok(got, f, oracle.reduce_f32(f, "sum"))
    assert same(tk.reduce(df, "max").item(), oracle.reduce_f32(f, "max"))
    assert same(tk.reduce(df, "min").item(), oracle.reduce_f32(f, "min"))
