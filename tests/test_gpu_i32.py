"""int32 TopK on the GPU, through the C ABI, against the CPU oracle.

Bit-exact: the output is an int32 multiset sorted descending, so the GPU's
k values must equal the oracle's element by element.  Small and medium sizes
are compared with the full oracle (std::sort); the 1e8 and 1e9 workloads are
checked with the oracle's exact one-pass checker (which the CPU tests pin
against the full oracle), and the 1e8 one also with the full oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

INT_MIN, INT_MAX = -(2**31), 2**31 - 1


@pytest.fixture(scope="module")
def tk():
    import topk_selection_gb300

    yield topk_selection_gb300
    # No kernel of this module gave up on a bounded device-side wait.
    topk_selection_gb300.check_stream()


def gpu_topk(tk, x_np, k, offset=0, stream=None):
    """Copy x to the device at an element offset (so the base pointer can be
    misaligned to 16 bytes) and run topk_i32 there."""
    buf = torch.empty(x_np.size + offset, dtype=torch.int32, device="cuda")
    view = buf[offset:]
    view.copy_(torch.from_numpy(x_np))
    out = tk.topk_i32(view, k, stream=stream)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def make(kind, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "uniform":
        return synth.i32_uniform(n, seed)
    if kind == "ascending":
        return np.arange(n, dtype=np.int64).astype(np.int32)
    if kind == "descending":
        return np.arange(n, 0, -1, dtype=np.int64).astype(np.int32)
    if kind == "equal":
        return np.full(n, 7, dtype=np.int32)
    if kind == "int_min":
        return np.full(n, INT_MIN, dtype=np.int32)
    if kind == "negative":
        return rng.integers(INT_MIN, 0, size=n, dtype=np.int64).astype(np.int32)
    if kind == "dups":
        return rng.integers(0, 1000, size=n).astype(np.int32)
    if kind == "few":
        return rng.choice(np.array([INT_MIN, -1, 0, 1, INT_MAX], dtype=np.int32), size=n)
    if kind == "int_max_heavy":
        x = rng.integers(INT_MIN, INT_MAX, size=n, dtype=np.int64).astype(np.int32)
        x[rng.random(n) < 0.3] = INT_MAX
        return x
    if kind == "sawtooth":
        return (np.arange(n, dtype=np.int64) % 1009).astype(np.int32)
    raise KeyError(kind)


KINDS = ["uniform", "ascending", "descending", "equal", "int_min", "negative", "dups", "few",
         "int_max_heavy", "sawtooth"]
SIZES = [1, 2, 3, 4, 5, 7, 31, 33, 127, 129, 1023, 1025, 4095, 4097, 65537, 300_007]
KS = [1, 2, 20, 32, 33, 64, 65, 100, 128, 129, 1000, 1024]


@pytest.mark.parametrize("kind", KINDS)
def test_edge_sizes_and_ks(tk, kind):
    for i, n in enumerate(SIZES):
        x = make(kind, n, seed=n)
        for k in KS:
            if k > n:
                continue
            got = gpu_topk(tk, x, k)
            exp = oracle.topk_i32(x, k)
            assert np.array_equal(got, exp), (kind, n, k, got[:8], exp[:8])


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_base(tk, offset):
    for n in (5, 6, 7, 1029, 262_147):
        x = make("uniform", n, seed=offset)
        for k in (1, 20, 100):
            if k <= n:
                assert np.array_equal(gpu_topk(tk, x, k, offset=offset), oracle.topk_i32(x, k))


def test_many_tiles_ragged_tail(tk):
    # Several tiles per warp and a last tile that is only partly filled.
    for n in (2_000_003, 4_194_305):
        x = make("uniform", n, seed=n)
        for k in (1, 20, 64, 100, 128):
            assert np.array_equal(gpu_topk(tk, x, k), oracle.topk_i32(x, k)), (n, k)


@pytest.mark.parametrize("cap", [2, 64])
def test_second_stage_radix_select_path(tk, cap):
    # With the second stage's shared list capped, more candidates exceed the
    # final threshold than fit, and the exact k-th value is found by radix
    # select over the candidates first.
    tk.set_option(tk.OPT_STAGE2_CAP, cap)
    try:
        for kind, n in (("uniform", 2_000_003), ("dups", 1_000_001), ("negative", 700_001), ("few", 90_001),
                        ("int_max_heavy", 500_009), ("sawtooth", 3_000_017)):
            x = make(kind, n, seed=n)
            for k in (1, 20, 64, 100, 128, 500):
                assert np.array_equal(gpu_topk(tk, x, k), oracle.topk_i32(x, k)), (kind, n, k, cap)
    finally:
        tk.set_option(tk.OPT_STAGE2_CAP, 0)


@pytest.mark.parametrize("kind,n", [("uniform", 1_000_003), ("dups", 2_000_003), ("few", 2_000_003),
                                    ("ascending", 3_000_000), ("descending", 999_999), ("equal", 400_000),
                                    ("int_min", 300_007), ("negative", 1_500_001), ("sawtooth", 1_234_567),
                                    ("int_max_heavy", 700_001)])
def test_large_k_radix_select(tk, kind, n):
    # k > 128: sampled threshold, one filter pass, cluster select and sort.
    x = make(kind, n, seed=n)
    for k in (129, 1000, 4096, 32768):
        assert np.array_equal(gpu_topk(tk, x, k), oracle.topk_i32(x, k)), (kind, n, k)


@pytest.mark.parametrize("kind,n", [("uniform", 1_000_003), ("dups", 2_000_003), ("few", 700_001),
                                    ("ascending", 3_000_000), ("negative", 1_500_001), ("sawtooth", 1_234_567),
                                    ("int_max_heavy", 700_001), ("equal", 400_000)])
def test_large_k_exact_passes(tk, kind, n):
    # The sampled threshold is only a shortcut: when it misleads the filter,
    # exact radix passes take over.  Sample rank 1 puts the threshold at the
    # sample's maximum, so the filter keeps fewer than k keys; a buffer capped
    # at k (option value 1) makes the filter overflow and makes the second
    # exact pass histogram instead of collect.  Sample rank 2000 leaves tens
    # of thousands of candidates, so that the final of a small k runs on the
    # whole cluster instead of one CTA.
    x = make(kind, n, seed=n + 1)
    try:
        for rank, cap in ((1, 0), (1, 1), (0, 1), (0, 6000), (2000, 0)):
            tk.set_option(tk.OPT_RADIX_SAMPLE_RANK, rank)
            tk.set_option(tk.OPT_RADIX_CAP, cap)
            for k in (129, 1000, 5000):
                assert np.array_equal(gpu_topk(tk, x, k), oracle.topk_i32(x, k)), (kind, n, k, rank, cap)
    finally:
        tk.set_option(tk.OPT_RADIX_SAMPLE_RANK, 0)
        tk.set_option(tk.OPT_RADIX_CAP, 0)


def test_large_k_cluster_only_sizes(tk):
    # n up to 2^18 runs the single cluster launch on the input itself.
    for n, k in ((262_144, 32_768), (262_144, 129), (262_145, 32_768), (200_000, 200_000 // 7), (4096, 4096)):
        for kind in ("uniform", "ascending", "dups", "equal"):
            x = make(kind, n, seed=n + k)
            assert np.array_equal(gpu_topk(tk, x, k), oracle.topk_i32(x, k)), (kind, n, k)


def test_large_k_full_sort_and_edges(tk):
    for n, k in ((129, 129), (32768, 32768), (40000, 32768), (1025, 1000), (5000, 4097)):
        x = make("uniform", n, seed=n + k)
        assert np.array_equal(gpu_topk(tk, x, k), oracle.topk_i32(x, k)), (n, k)
    x = make("uniform", 300_007, seed=5)
    for offset in (1, 2, 3):
        assert np.array_equal(gpu_topk(tk, x, 777, offset=offset), oracle.topk_i32(x, 777))


def test_plans_alternate_on_one_workspace(tk):
    # The streaming plan (k <= 128) and the radix plan (k > 128) share the
    # workspace of a stream; each must leave it as the other expects.
    x = make("uniform", 2_000_003, seed=9)
    y = make("dups", 1_000_003, seed=10)
    for k in (20, 500, 64, 2000, 1, 129, 128):
        for v in (x, y):
            assert np.array_equal(gpu_topk(tk, v, k), oracle.topk_i32(v, k)), k


def test_back_to_back_calls_reset_state(tk):
    # The control words are reset by each launch: a large threshold left by a
    # call must not leak into the next call on the same stream.
    big = np.full(500_000, INT_MAX, dtype=np.int32)
    small = make("negative", 400_000, seed=3)
    s = torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(s):
            a = gpu_topk(tk, big, 20, stream=s)
            b = gpu_topk(tk, small, 20, stream=s)
        assert np.array_equal(a, oracle.topk_i32(big, 20))
        assert np.array_equal(b, oracle.topk_i32(small, 20))


def test_chained_calls_read_the_previous_output(tk):
    # Back-to-back launches on one stream may overlap (the next starts
    # streaming while the previous finishes), except when the next call's
    # input is the previous call's output: that chain must see the finished
    # values.
    x = synth.i32_uniform(5_000_000, 31)
    d = torch.from_numpy(x).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(5):
            a = tk.topk_i32(d, 128, stream=s)
            b = tk.topk_i32(a, 20, stream=s)      # input = the previous output
            c = tk.topk_i32(d, 64, stream=s)      # independent input: may overlap b
            e = tk.topk_i32(c, 1, stream=s)
    s.synchronize()
    exp = oracle.topk_i32(x, 128)
    assert np.array_equal(a.cpu().numpy(), exp)
    assert np.array_equal(b.cpu().numpy(), exp[:20])
    assert np.array_equal(c.cpu().numpy(), exp[:64])
    assert e.cpu().numpy()[0] == exp[0]


def test_chains_through_the_large_k_plan(tk):
    # The large-k kernels release their successors early as well: a
    # streaming call on a large-k call's output must still see it finished,
    # and the other way round.
    x = synth.i32_uniform(4_000_000, 32)
    d = torch.from_numpy(x).cuda()
    s = torch.cuda.Stream()
    exp = oracle.topk_i32(x, 5000)
    with torch.cuda.stream(s):
        for _ in range(4):
            a = tk.topk_i32(d, 5000, stream=s)    # large-k plan
            b = tk.topk_i32(a, 100, stream=s)     # streaming, input = a
            c = tk.topk_i32(d, 120, stream=s)     # streaming, independent
            f = tk.topk_i32(c, 110, stream=s)     # streaming on c
            g = tk.topk_i32(a, 4000, stream=s)    # large-k on a
            h = tk.topk_i32(g, 7, stream=s)       # streaming on g
    s.synchronize()
    assert np.array_equal(a.cpu().numpy(), exp)
    assert np.array_equal(b.cpu().numpy(), exp[:100])
    assert np.array_equal(c.cpu().numpy(), exp[:120])
    assert np.array_equal(f.cpu().numpy(), exp[:110])
    assert np.array_equal(g.cpu().numpy(), exp[:4000])
    assert np.array_equal(h.cpu().numpy(), exp[:7])


def test_many_back_to_back_calls(tk):
    # A long run of overlapping launches on one stream, inputs and outputs
    # distinct: every result must match.
    xs = [synth.i32_uniform(3_000_000 + 17 * i, 40 + i) for i in range(4)]
    ds = [torch.from_numpy(x).cuda() for x in xs]
    outs = []
    for rep in range(50):
        for i, d in enumerate(ds):
            outs.append((i, tk.topk_i32(d, (20, 1, 100, 64)[i])))
    torch.cuda.synchronize()
    exps = [oracle.topk_i32(x, k) for x, k in zip(xs, (20, 1, 100, 64))]
    for i, o in outs:
        assert np.array_equal(o.cpu().numpy(), exps[i])


def test_non_default_stream_in_flight(tk):
    x = synth.i32_uniform(3_000_000, 11)
    d = torch.from_numpy(x).cuda()
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for k in (1, 20, 100):
            outs.append((k, tk.topk_i32(d, k)))
    s.synchronize()
    for k, o in outs:
        assert np.array_equal(o.cpu().numpy(), oracle.topk_i32(x, k))


def test_host_buffers(tk):
    # CPU tensors: the library stages them through device memory itself.
    x = synth.i32_uniform(1_000_003, 21)
    xt = torch.from_numpy(x)
    for pin in (False, True):
        src = xt.pin_memory() if pin else xt
        out = torch.empty(20, dtype=torch.int32, pin_memory=pin)
        tk.topk_i32(src, 20, out=out)
        assert np.array_equal(out.numpy(), oracle.topk_i32(x, 20))


def test_workload_2p20(tk):
    x = synth.i32_workload("i32_uniform_2p20")
    assert np.array_equal(gpu_topk(tk, x, 20), oracle.topk_i32(x, 20))


def test_workload_1e7(tk):
    x = synth.i32_workload("i32_uniform_1e7")
    for k in (20, 100):
        assert np.array_equal(gpu_topk(tk, x, k), oracle.topk_i32(x, k))


def test_workload_1e8(tk):
    x = synth.i32_workload("i32_uniform_1e8")
    d = torch.from_numpy(x).cuda()
    for k in (20, 1):
        got = tk.topk_i32(d, k).cpu().numpy()
        assert oracle.check_topk_i32(x, k, got)
        if k == 20:
            assert np.array_equal(got, oracle.topk_i32(x, k))
        else:
            assert got[0] == x.max()
    del d


@pytest.mark.parametrize("name", ["i32_uniform_1e9", "i32_ascending_1e9", "i32_dup1000_1e9"])
def test_workload_1e9(tk, name):
    x = synth.i32_workload(name)
    d = torch.from_numpy(x).cuda()
    got = tk.topk_i32(d, 20).cpu().numpy()
    del d
    torch.cuda.empty_cache()
    assert oracle.check_topk_i32(x, 20, got), (name, got)
    if name == "i32_ascending_1e9":
        assert got.tolist() == list(range(10**9 - 1, 10**9 - 21, -1))
    if name == "i32_dup1000_1e9":
        assert got.tolist() == [999] * 20


@pytest.mark.parametrize("static", [1, 51, 101])
def test_tile_schedules(tk, static):
    # The streaming plan shares out part of the tiles up front and lets warps
    # claim the rest from 64 counters; all-claimed (1), half (51) and
    # all-static (101) schedules must give the same exact result, including
    # sizes with fewer dynamic tiles than counters and a ragged last tile.
    tk.set_option(tk.OPT_STREAM_STATIC, static)
    try:
        for kind, n in (("uniform", 4_194_305), ("ascending", 3_000_001), ("dups", 1_000_003),
                        ("uniform", 65_537), ("few", 300_007), ("uniform", 25_000_003)):
            x = make(kind, n, seed=n + static)
            for k in (1, 20, 64, 128):
                assert np.array_equal(gpu_topk(tk, x, k), oracle.topk_i32(x, k)), (kind, n, k, static)
        # Back-to-back calls on one stream reuse the claim counters.
        x = make("uniform", 9_000_011, seed=5)
        d = torch.from_numpy(x).cuda()
        outs = [tk.topk_i32(d, 20) for _ in range(6)]
        exp = oracle.topk_i32(x, 20)
        for o in outs:
            assert np.array_equal(o.cpu().numpy(), exp)
    finally:
        tk.set_option(tk.OPT_STREAM_STATIC, 0)


def test_few_blocks_many_k(tk):
    # Inputs small enough that the grid has fewer blocks than k: the second
    # stage bounds the answer by the k-th largest tile maximum.
    for kind in KINDS:
        for n in (40_000, 100_003, 300_007, 900_001):
            x = make(kind, n, seed=n + 3)
            for k in (65, 100, 128):
                assert np.array_equal(gpu_topk(tk, x, k), oracle.topk_i32(x, k)), (kind, n, k)


def test_early_start_record(tk):
    # A streaming call may start early only after a releasing launch whose
    # output it does not read (topk_last_launch_early reports the decision).
    s = torch.cuda.Stream()
    x = torch.from_numpy(synth.i32_uniform(2_000_003, 9)).cuda()
    with torch.cuda.stream(s):
        a = tk.topk_i32(x, 64, stream=s)          # first call on this stream
        assert not tk.last_launch_early()
        tk.topk_i32(x, 20, stream=s)              # after a releasing launch, independent input
        assert tk.last_launch_early()
        b = tk.topk_i32(a, 10, stream=s)          # reads an older call's output, finished before the last one released
        assert tk.last_launch_early()
        tk.topk_i32(b, 5, stream=s)               # reads the previous call's output
        assert not tk.last_launch_early()
        tk.reduce(x, "sum", stream=s)             # does not release
        tk.topk_i32(x, 20, stream=s)
        assert not tk.last_launch_early()
    s.synchronize()
