"""uint32 and float32 keys on the GPU (topk_u32, topk_f32), through the C ABI,
against the CPU oracle.

Bit-exact: the outputs are key multisets sorted descending, in unsigned
order (uint32) or IEEE 754 totalOrder (float32, the order of the radix sort
page's float bit transform), so the GPU's k words must equal the oracle's
word by word.  Both plans are covered: the streaming plan (k <= 128) and the
radix-select plan (larger k), on inputs full of the values that order
differently from int32: words above 2^31 - 1, negative floats, -0.0 / +0.0,
infinities, NaNs of both signs with different payloads, denormals.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

SPECIAL_BITS = np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0x7FC00001, 0xFFC00000,
                         0xFFC00001, 0x7F800001, 0x00000001, 0x80000001, 0x3F800000, 0xBF800000, 0x7F7FFFFF,
                         0xFF7FFFFF], dtype=np.uint32)


@pytest.fixture(scope="module")
def tk():
    import topk_selection_gb300

    yield topk_selection_gb300
    topk_selection_gb300.check_stream()


def f32_input(kind, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return synth.f32_normal(n, seed)
    if kind == "specials":
        x = synth.f32_normal(n, seed).view(np.uint32).copy()
        pick = rng.random(n) < 0.2
        x[pick] = rng.choice(SPECIAL_BITS, size=int(pick.sum()))
        return x.view(np.float32)
    if kind == "bits":  # every bit pattern equally likely: half negative, some NaN
        return synth.i32_uniform(n, seed).view(np.float32)
    if kind == "zeros":
        return rng.choice(np.array([0x00000000, 0x80000000], dtype=np.uint32), size=n).view(np.float32)
    if kind == "negative":
        return -np.abs(synth.f32_normal(n, seed))
    if kind == "dups":
        return (rng.integers(-50, 50, size=n) * 0.25).astype(np.float32)
    if kind == "nan_heavy":
        x = rng.choice(SPECIAL_BITS[4:9], size=n).astype(np.uint32)
        return x.view(np.float32)
    raise KeyError(kind)


def u32_input(kind, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "uniform":
        return synth.i32_uniform(n, seed).view(np.uint32)
    if kind == "high":  # all above 2^31 - 1: int32 order would reverse them
        return (synth.i32_uniform(n, seed).view(np.uint32) | np.uint32(0x80000000))
    if kind == "mixed_top":
        return rng.choice(np.array([0, 1, 2**31 - 1, 2**31, 2**32 - 1], dtype=np.uint32), size=n)
    if kind == "ascending":
        return np.arange(n, dtype=np.uint64).astype(np.uint32) + np.uint32(2**31 - n // 2)
    raise KeyError(kind)


def run_f32(tk, x, k, offset=0):
    buf = torch.empty(x.size + offset, dtype=torch.float32, device="cuda")
    view = buf[offset:]
    view.copy_(torch.from_numpy(x))
    out = tk.topk_f32(view, k)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint32)


def run_u32(tk, x, k, offset=0):
    buf = torch.empty(x.size + offset, dtype=torch.int32, device="cuda")
    view = buf[offset:]
    view.copy_(torch.from_numpy(x.view(np.int32)))
    out = tk.topk_u32(view, k)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint32)


F32_KINDS = ["normal", "specials", "bits", "zeros", "negative", "dups", "nan_heavy"]
U32_KINDS = ["uniform", "high", "mixed_top", "ascending"]
SIZES = [1, 5, 33, 1025, 65_537, 300_007, 2_000_003]
KS = [1, 2, 20, 64, 100, 128, 129, 1000, 4096]


@pytest.mark.parametrize("kind", F32_KINDS)
def test_f32_sizes_and_ks(tk, kind):
    for n in SIZES:
        x = f32_input(kind, n, seed=n)
        exp_all = oracle.topk_f32(x, min(n, max(KS)))
        for k in KS:
            if k > n:
                continue
            got = run_f32(tk, x, k)
            assert np.array_equal(got, exp_all[:k].view(np.uint32)), (kind, n, k)


@pytest.mark.parametrize("kind", U32_KINDS)
def test_u32_sizes_and_ks(tk, kind):
    for n in SIZES:
        x = u32_input(kind, n, seed=n)
        exp_all = oracle.topk_u32(x, min(n, max(KS)))
        for k in KS:
            if k > n:
                continue
            assert np.array_equal(run_u32(tk, x, k), exp_all[:k]), (kind, n, k)


@pytest.mark.parametrize("offset", [1, 3])
def test_misaligned(tk, offset):
    for n in (7, 4099, 1_000_003):
        xf = f32_input("specials", n, seed=offset)
        xu = u32_input("uniform", n, seed=offset)
        for k in (1, 20, 128, 500):
            if k <= n:
                assert np.array_equal(run_f32(tk, xf, k, offset), oracle.topk_f32(xf, k).view(np.uint32))
                assert np.array_equal(run_u32(tk, xu, k, offset), oracle.topk_u32(xu, k))


def test_large_inputs(tk):
    # The 1e8-scale shapes of the TopK pages' table, both plans.
    n = 50_000_003
    xf = f32_input("specials", n, seed=9)
    exp = oracle.topk_f32(xf, 32768).view(np.uint32)
    for k in (1, 20, 128, 1000, 32768):
        assert np.array_equal(run_f32(tk, xf, k), exp[:k]), k
    xu = u32_input("uniform", n, seed=10)
    expu = oracle.topk_u32(xu, 32768)
    for k in (20, 100, 129, 32768):
        assert np.array_equal(run_u32(tk, xu, k), expu[:k]), k


def test_exact_passes_with_float_keys(tk):
    # Force the large-k plan's exact passes (sample threshold at its top) on
    # float keys, so that the exact histograms see the transformed order too.
    tk.set_option(tk.OPT_RADIX_SAMPLE_RANK, 1)
    try:
        for kind in ("specials", "bits", "zeros"):
            x = f32_input(kind, 3_000_017, seed=4)
            for k in (129, 2000):
                assert np.array_equal(run_f32(tk, x, k), oracle.topk_f32(x, k).view(np.uint32)), (kind, k)
        xu = u32_input("high", 3_000_017, seed=5)
        assert np.array_equal(run_u32(tk, xu, 700), oracle.topk_u32(xu, 700))
    finally:
        tk.set_option(tk.OPT_RADIX_SAMPLE_RANK, 0)


def test_kinds_share_a_stream(tk):
    # Back to back on one stream and one workspace: int32, uint32 and float32
    # calls of both plans, each on the previous one's output or independent.
    xf = f32_input("specials", 4_000_037, seed=21)
    xu = u32_input("high", 4_000_037, seed=22)
    df, du = torch.from_numpy(xf).cuda(), torch.from_numpy(xu.view(np.int32)).cuda()
    a = tk.topk_f32(df, 3000)
    b = tk.topk_u32(du, 64)
    c = tk.topk_f32(a, 20)
    d = tk.topk_i32(du, 100)
    e = tk.topk_u32(b, 10)
    torch.cuda.synchronize()
    ef = oracle.topk_f32(xf, 3000).view(np.uint32)
    eu = oracle.topk_u32(xu, 64)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ef)
    assert np.array_equal(b.cpu().numpy().view(np.uint32), eu)
    assert np.array_equal(c.cpu().numpy().view(np.uint32), ef[:20])
    assert np.array_equal(d.cpu().numpy(), oracle.topk_i32(xu.view(np.int32), 100))
    assert np.array_equal(e.cpu().numpy().view(np.uint32), eu[:10])


@pytest.mark.parametrize("n", [131_072, 200_003, 3_000_017, 20_000_003])
def test_k_beyond_32768(tk, n):
    # k above the range plan's 32768: the cluster leaves the answer unordered
    # and the LSD radix sort orders it (n <= 2^18 takes the one-cluster form).
    ks = [k for k in (32_769, 65_536, 100_000, 131_072) if k <= n]
    xi = synth.i32_mod(n, n, 1000) if n == 200_003 else synth.i32_uniform(n, n)
    xf = f32_input("specials", n, seed=n + 1)
    xu = u32_input("high", n, seed=n + 2)
    ei = oracle.topk_i32(xi, max(ks))
    ef = oracle.topk_f32(xf, max(ks)).view(np.uint32)
    eu = oracle.topk_u32(xu, max(ks))
    for k in ks:
        gi = tk.topk_i32(torch.from_numpy(xi).cuda(), k).cpu().numpy()
        assert np.array_equal(gi, ei[:k]), ("i32", n, k)
        assert np.array_equal(run_f32(tk, xf, k), ef[:k]), ("f32", n, k)
        assert np.array_equal(run_u32(tk, xu, k), eu[:k]), ("u32", n, k)


def test_k_beyond_32768_exact_passes_and_ties(tk):
    # The big-k form after the exact passes (sample rank forced to 1), on
    # heavy ties (values in [0, 1000): the k-th value repeats ~3000 times) and
    # on all-equal input.
    tk.set_option(tk.OPT_RADIX_SAMPLE_RANK, 1)
    try:
        x = synth.i32_mod(3_000_017, 8, 1000)
        d = torch.from_numpy(x).cuda()
        for k in (40_000, 131_072):
            assert np.array_equal(tk.topk_i32(d, k).cpu().numpy(), oracle.topk_i32(x, k)), k
    finally:
        tk.set_option(tk.OPT_RADIX_SAMPLE_RANK, 0)
    same = np.full(1_000_000, -3, dtype=np.int32)
    assert np.array_equal(tk.topk_i32(torch.from_numpy(same).cuda(), 100_000).cpu().numpy(),
                          np.full(100_000, -3, dtype=np.int32))
    # back to back with the streaming and range plans on one stream
    x = synth.i32_uniform(5_000_011, 12)
    d = torch.from_numpy(x).cuda()
    outs = [tk.topk_i32(d, k) for k in (100_000, 20, 5000, 131_072, 128)]
    exp = oracle.topk_i32(x, 131_072)
    for o in outs:
        assert np.array_equal(o.cpu().numpy(), exp[:o.numel()]), o.numel()
