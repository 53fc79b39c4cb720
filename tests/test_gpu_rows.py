"""Row TopK with indices on the GPU, through the C ABI, against the oracle.

Bit-exact: column indices must equal the oracle's (value descending, lower
column first among equal values) and the values must carry the input's bits.
The 4096 x 32768 workload is compared with the oracle on a spread of sampled
rows, and every row is checked for the properties that pin the answer (the
k-th entry is beaten by exactly k-1 elements of its row, values are the
input's bits at the returned columns, columns are distinct and ordered).
"""
import math
import struct

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


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def gpu_rows(tk, x, k, col_offset=0):
    rows, cols = x.shape
    if col_offset:
        # Rows placed at an element offset so row starts are not 16-byte aligned.
        buf = torch.empty(rows * cols + col_offset, dtype=torch.float32, device="cuda")
        dx = buf[col_offset:].view(rows, cols)
        dx.copy_(torch.from_numpy(x))
    else:
        dx = torch.from_numpy(x).cuda()
    v, i = tk.topk_rows_f32(dx, k)
    torch.cuda.synchronize()
    return v.cpu().numpy(), i.cpu().numpy()


def assert_rows_equal(tk, x, k, col_offset=0):
    v, i = gpu_rows(tk, x, k, col_offset)
    ev, ei = oracle.topk_rows_f32(x, k)
    bad = np.nonzero(~np.all(i == ei, axis=1))[0]
    assert bad.size == 0, (k, x.shape, bad[:5], i[bad[0]][:8], ei[bad[0]][:8])
    assert np.array_equal(bits(v), bits(ev)), (k, x.shape)


SPECIAL = np.array([math.nan, -math.inf, math.inf, -0.0, 0.0, 1.0, -1.0, 3.4e38, -3.4e38, 1e-45, -1e-45],
                   dtype=np.float32)


@pytest.mark.parametrize("cols", [1, 2, 3, 4, 5, 31, 33, 127, 1024, 1025, 4099, 32768])
def test_shapes_and_ks(tk, cols):
    rng = np.random.default_rng(cols)
    rows = 37
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    x[1] = 2.0                              # a row of equal values
    x[2] = np.round(x[2] * 2) / 2           # many ties
    x[3] = SPECIAL[rng.integers(0, SPECIAL.size, cols)]
    x[4] = -np.abs(x[4])                    # all negative
    for k in (1, 2, 7, 32, 33, 64, 100, 128, 129, 500, 1024):
        if k <= cols:
            assert_rows_equal(tk, x, k)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_rows(tk, offset):
    rng = np.random.default_rng(offset)
    x = rng.standard_normal((19, 2051)).astype(np.float32)
    for k in (1, 64, 129):
        assert_rows_equal(tk, x, k, col_offset=offset)


def test_signed_zero_and_nan_payload(tk):
    neg_nan = struct.unpack("<f", struct.pack("<I", 0xFFC12345))[0]
    x = np.zeros((4, 64), dtype=np.float32)
    x[0, ::2] = -0.0
    x[1, 5] = neg_nan
    x[1, 9] = math.nan
    x[2, :] = -math.inf
    x[3, 40:] = math.inf
    for k in (1, 3, 64):
        assert_rows_equal(tk, x, k)
    v, i = gpu_rows(tk, x, 2)
    assert i[1].tolist() == [5, 9]
    assert bits(v[1])[0] == 0xFFC12345


def test_tied_rows_small(tk):
    x = synth.f32_rows_tied(128, 4096, 5)
    for k in (1, 40, 41, 64, 128):
        assert_rows_equal(tk, x, k)


def test_host_buffers(tk):
    x = synth.f32_rows_tied(33, 1000, 7)
    ev, ei = oracle.topk_rows_f32(x, 64)
    v, i = tk.topk_rows_f32(torch.from_numpy(x), 64)
    assert np.array_equal(i.numpy(), ei)
    assert np.array_equal(bits(v.numpy()), bits(ev))


def check_all_rows(x, k, v, i):
    rows, cols = x.shape
    # values are the input's bits at the returned columns
    assert np.array_equal(bits(v), bits(np.take_along_axis(x, i.astype(np.int64), axis=1)))
    # columns are distinct per row
    s = np.sort(i, axis=1)
    assert np.all(s[:, 1:] != s[:, :-1])
    # order: value descending, lower column first among equal values (no NaN here)
    a, b = v[:, :-1], v[:, 1:]
    assert np.all((a > b) | ((a == b) & (i[:, :-1] < i[:, 1:])))
    # exactly k-1 elements of the row beat the k-th entry
    kv, ki = v[:, -1:], i[:, -1:]
    col = np.arange(cols)[None, :]
    beat = (x > kv) | ((x == kv) & (col < ki))
    assert np.all(beat.sum(axis=1) == k - 1)


@pytest.mark.parametrize("tied", [True, False])
def test_workload_4096x32768(tk, tied):
    w = synth.ROWS_WORKLOAD
    rows, cols, k = w["rows"], w["cols"], w["k"]
    x = synth.f32_rows_tied(rows, cols, w["seed"], w["tie_frac"]) if tied else \
        synth.f32_rows_normal(rows, cols, w["seed"])
    v, i = gpu_rows(tk, x, k)
    sample = np.unique(np.linspace(0, rows - 1, 256).astype(np.int64))
    ev, ei = oracle.topk_rows_f32(x[sample], k)
    assert np.array_equal(i[sample], ei)
    assert np.array_equal(bits(v[sample]), bits(ev))
    for lo in range(0, rows, 512):
        check_all_rows(x[lo:lo + 512], k, v[lo:lo + 512], i[lo:lo + 512])


def special_rows(rows, cols, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    special = [
        lambda r: np.full(cols, 1.5, np.float32),                 # one value: every column ties
        lambda r: np.round(r * 4) / 4,                            # many ties
        lambda r: SPECIAL[rng.integers(0, SPECIAL.size, cols)],
        lambda r: -np.abs(r),
        lambda r: np.concatenate([r[:-5], np.full(5, 9.0, np.float32)]),   # the best values at the end
        lambda r: np.concatenate([np.full(5, 9.0, np.float32), r[5:]]),    # and at the start
    ]
    for i, f in enumerate(special[:rows]):
        x[i] = f(x[i])
    if rows > len(special):
        z = np.full(cols, -0.0, np.float32)
        z[rng.integers(0, cols, 40)] = 0.0
        x[len(special)] = z
    return x


def test_long_rows_with_specials(tk):
    x = special_rows(11, 50_003, 1)
    for k in (1, 20, 33, 64, 100, 128, 129, 300, 1024):
        assert_rows_equal(tk, x, k)
    assert_rows_equal(tk, x[:, :49_997], 64, col_offset=3)
    assert_rows_equal(tk, x[:, :49_997], 777, col_offset=1)


@pytest.mark.parametrize("k", [256, 1024])
@pytest.mark.parametrize("tied", [True, False])
def test_workload_shape_large_k(tk, k, tied):
    # k > 128: one block per row with a shared candidate buffer.
    w = synth.ROWS_WORKLOAD
    rows, cols = w["rows"], w["cols"]
    x = synth.f32_rows_tied(rows, cols, w["seed"], w["tie_frac"]) if tied else \
        synth.f32_rows_normal(rows, cols, w["seed"])
    v, i = gpu_rows(tk, x, k)
    sample = np.unique(np.linspace(0, rows - 1, 64).astype(np.int64))
    ev, ei = oracle.topk_rows_f32(x[sample], k)
    assert np.array_equal(i[sample], ei)
    assert np.array_equal(bits(v[sample]), bits(ev))
    for lo in range(0, rows, 512):
        check_all_rows(x[lo:lo + 512], k, v[lo:lo + 512], i[lo:lo + 512])


def test_few_long_rows(tk):
    # 1.5M columns: hundreds of rounds and many cuts per row for k > 128;
    # row 1 is all equal (the cuts separate keys by column alone).
    x = synth.f32_rows_tied(3, 1_500_001, 11)
    x[1] = np.float32(0.25)
    for k in (1, 64, 128, 129, 1024):
        assert_rows_equal(tk, x, k)


def test_shapes_back_to_back(tk):
    # Different shapes one after the other on one stream.
    shapes = [(7, 100_000, 64), (5000, 800, 10), (64, 32768, 128), (1, 300_000, 1), (4500, 2000, 32)]
    data = {sh: special_rows(sh[0], sh[1], sum(sh)) for sh in shapes}
    expect = {sh: oracle.topk_rows_f32(data[sh], sh[2]) for sh in shapes}
    dev = {sh: torch.from_numpy(data[sh]).cuda() for sh in shapes}
    for rep in range(2):
        outs = [(sh, tk.topk_rows_f32(dev[sh], sh[2])) for sh in shapes]
        torch.cuda.synchronize()
        for sh, (v, i) in outs:
            ev, ei = expect[sh]
            assert np.array_equal(i.cpu().numpy(), ei), (rep, sh)
            assert np.array_equal(bits(v.cpu().numpy()), bits(ev)), (rep, sh)


def test_chained_and_overlapping_calls(tk):
    # Row calls (k <= 128) may start while the previous launch on the stream
    # finishes, except when their input is that launch's output; int32 calls
    # share the rule.
    x = special_rows(300, 20_000, 9)
    y = synth.f32_rows_tied(200, 9000, 10)
    dx, dy = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    ev1, ei1 = oracle.topk_rows_f32(x, 64)
    ev2, ei2 = oracle.topk_rows_f32(ev1, 8)
    evy, eiy = oracle.topk_rows_f32(y, 32)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(4):
            v1, i1 = tk.topk_rows_f32(dx, 64, stream=s)
            v2, i2 = tk.topk_rows_f32(v1, 8, stream=s)       # input = previous vals
            vy, iy = tk.topk_rows_f32(dy, 32, stream=s)      # independent
            t = tk.topk_i32(iy.view(-1), 5, stream=s)        # int32 on the previous idx
            v3, i3 = tk.topk_rows_f32(dy, 32, stream=s)      # after an int32 call
    s.synchronize()
    assert np.array_equal(i1.cpu().numpy(), ei1) and np.array_equal(bits(v1.cpu().numpy()), bits(ev1))
    assert np.array_equal(i2.cpu().numpy(), ei2) and np.array_equal(bits(v2.cpu().numpy()), bits(ev2))
    assert np.array_equal(iy.cpu().numpy(), eiy) and np.array_equal(bits(vy.cpu().numpy()), bits(evy))
    assert np.array_equal(t.cpu().numpy(), oracle.topk_i32(eiy.reshape(-1).astype(np.int32), 5))
    assert np.array_equal(i3.cpu().numpy(), eiy) and np.array_equal(bits(v3.cpu().numpy()), bits(evy))


@pytest.mark.parametrize("cols", [65_536, 65_537])
def test_select_deeper_levels_and_kernel_boundary(tk, cols):
    # 128 < k <= 1024 on rows up to 65536 columns is a per-row radix select
    # whose first 11-bit bucket must hold at most 4096 candidates; these rows
    # make it hold more, so further digit levels (score bits, then column
    # bits) decide.  65537 columns take the streamed kernel instead.
    rng = np.random.default_rng(cols)
    x = rng.standard_normal((8, cols)).astype(np.float32)
    x[0] = rng.uniform(1.0, 1.25, cols).astype(np.float32)   # every key in one first-level bucket
    x[1] = np.float32(1.5)
    x[1, rng.choice(cols, 5000, replace=False)] = np.float32(7.0)  # 5000 copies of the largest value
    x[2] = np.float32(-3.0)                                   # all equal: columns alone decide
    x[3] = np.round(x[3] * 64) / 64                           # dense ties everywhere
    x[4, ::3] = np.nan                                        # NaN above +inf, equal among themselves
    for k in (129, 777, 1024):
        assert_rows_equal(tk, x, k)
