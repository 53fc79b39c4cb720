"""Score-keyed TopK with item ids and a keep filter on the GPU, through the C
ABI, against the oracle: scores (bits), items and count must be identical."""
import math

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


def run(tk, score, k, item=None, keep=None):
    d = torch.from_numpy(score).cuda()
    di = None if item is None else torch.from_numpy(item).cuda()
    dk = None if keep is None else torch.from_numpy(keep).cuda()
    s, i, c = tk.topk_items_f32(d, k, item=di, keep=dk)
    torch.cuda.synchronize()
    return s.cpu().numpy(), i.cpu().numpy(), int(c.item())


def check(tk, score, k, item=None, keep=None):
    gs, gi, gc = run(tk, score, k, item, keep)
    es, ei, ec = oracle.topk_items_f32(score, k, item=item, keep=keep)
    assert gc == ec, (score.size, k, gc, ec)
    bad = np.nonzero(gi != ei)[0]
    assert bad.size == 0, (score.size, k, bad[:5], gi[bad[:5]], ei[bad[:5]])
    assert np.array_equal(bits(gs), bits(es)), (score.size, k)


def make(kind, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return synth.f32_normal(n, seed)
    if kind == "ties":
        return (np.round(rng.standard_normal(n) * 4) / 4).astype(np.float32)
    if kind == "specials":
        pool = np.array([math.nan, math.inf, -math.inf, -0.0, 0.0, 1.0, -1.0, 2.0], dtype=np.float32)
        return pool[rng.integers(0, pool.size, n)]
    if kind == "equal":
        return np.full(n, 1.5, dtype=np.float32)
    raise KeyError(kind)


SIZES = [1, 2, 5, 33, 1000, 4097, 65537, 300_007]
KS = [1, 7, 64, 128, 129, 500, 1024]


@pytest.mark.parametrize("kind", ["normal", "ties", "specials", "equal"])
def test_sizes_ks_no_filter(tk, kind):
    for n in SIZES:
        x = make(kind, n, n)
        for k in KS:
            if k <= n:
                check(tk, x, k)


@pytest.mark.parametrize("frac", [0.5, 0.01, 0.0])
def test_filter_and_items(tk, frac):
    rng = np.random.default_rng(int(frac * 100) + 3)
    for n in (5, 1000, 65537, 300_007):
        x = make("ties", n, n + 1)
        keep = (rng.random(n) < frac).astype(np.uint8)
        items = rng.integers(-2**62, 2**62, size=n, dtype=np.int64)
        for k in (1, 64, 129, 1000):
            if k <= n:
                check(tk, x, k, item=items, keep=keep)


def test_filter_vector_and_scalar_paths(tk):
    # 16-byte-aligned arrays with n a multiple of 16 take the vector filter;
    # offset views or other n take the scalar one.  Both must agree with the
    # oracle.
    rng = np.random.default_rng(31)
    for n in (4096, 4097, 1_048_576, 1_048_577):
        x = make("ties", n, n)
        keep = (rng.random(n) < 0.4).astype(np.uint8)
        check(tk, x, 100, keep=keep)
        d = torch.empty(n + 1, dtype=torch.float32, device="cuda")
        d[1:].copy_(torch.from_numpy(x))
        kk = torch.empty(n + 1, dtype=torch.uint8, device="cuda")
        kk[1:].copy_(torch.from_numpy(keep))
        s_, i_, c_ = tk.topk_items_f32(d[1:], 100, keep=kk[1:])
        es, ei, ec = oracle.topk_items_f32(x, 100, keep=keep)
        assert int(c_.item()) == ec and np.array_equal(i_.cpu().numpy(), ei)
        assert np.array_equal(bits(s_.cpu().numpy()), bits(es))


def test_fewer_kept_than_k(tk):
    x = make("normal", 10_000, 5)
    keep = np.zeros(x.size, dtype=np.uint8)
    keep[[3, 500, 9999]] = 1
    check(tk, x, 64, keep=keep)
    keep[:] = 0
    check(tk, x, 10, keep=keep)
    keep[-1] = 1
    check(tk, x, 1, keep=keep)


def test_merge_is_topk_of_concatenation(tk):
    # Two TopK results merged: the TopK of their concatenated (score, item)
    # lists equals the TopK of the union of the inputs.
    a, b = make("ties", 200_000, 11), make("ties", 150_000, 12)
    ia = np.arange(a.size, dtype=np.int64)
    ib = np.arange(a.size, a.size + b.size, dtype=np.int64)
    k = 100
    sa, xa, _ = run(tk, a, k, item=ia)
    sb, xb, _ = run(tk, b, k, item=ib)
    ms, mi, _ = run(tk, np.concatenate([sa, sb]), k, item=np.concatenate([xa, xb]))
    es, ei, _ = oracle.topk_items_f32(np.concatenate([a, b]), k, item=np.concatenate([ia, ib]))
    assert np.array_equal(mi, ei) and np.array_equal(bits(ms), bits(es))


def test_large_filtered(tk):
    n = 20_000_000
    x = make("ties", n, 21)
    rng = np.random.default_rng(22)
    keep = (rng.random(n) < 0.3).astype(np.uint8)
    items = rng.integers(0, 2**40, size=n, dtype=np.int64)
    for k in (64, 1024):
        check(tk, x, k, item=items, keep=keep)
    check(tk, x, 128)



def run_views(tk, score, k, keep, item=None, score_off=0, keep_off=0):
    """topk_items_f32 on device views placed at element offsets."""
    n = score.size
    d = torch.empty(n + score_off, dtype=torch.float32, device="cuda")
    d[score_off:].copy_(torch.from_numpy(score))
    kk = torch.empty(n + keep_off, dtype=torch.uint8, device="cuda")
    kk[keep_off:].copy_(torch.from_numpy(keep))
    di = None if item is None else torch.from_numpy(item).cuda()
    s_, i_, c_ = tk.topk_items_f32(d[score_off:], k, item=di, keep=kk[keep_off:])
    torch.cuda.synchronize()
    return s_.cpu().numpy(), i_.cpu().numpy(), int(c_.item())


def check_views(tk, score, k, keep, item=None, score_off=0, keep_off=0):
    gs, gi, gc = run_views(tk, score, k, keep, item, score_off, keep_off)
    es, ei, ec = oracle.topk_items_f32(score, k, item=item, keep=keep)
    assert gc == ec, (score.size, k, score_off, keep_off, gc, ec)
    assert np.array_equal(gi, ei), (score.size, k, score_off, keep_off, gi[:5], ei[:5])
    assert np.array_equal(bits(gs), bits(es)), (score.size, k, score_off, keep_off)


@pytest.mark.parametrize("frac", [0.5, 0.01, 1.0, 0.0])
def test_filter_folded_into_first_level(tk, frac):
    # Large inputs with k <= 128 skip filtered positions inside the first
    # level: rows with fewer kept elements than k, kept -inf and NaN next to
    # larger filtered-out scores, and every offset pairing that keeps the
    # keep words aligned (and some that do not, which take the compaction).
    rng = np.random.default_rng(int(frac * 1000) + 77)
    n = (1 << 20) + 12_345
    x = make("specials", n, 7) if frac == 0.5 else make("ties", n, 8)
    keep = (rng.random(n) < frac).astype(np.uint8)
    keep[keep != 0] = rng.integers(1, 256, size=int(keep.sum()), dtype=np.uint8)  # any nonzero byte keeps
    items = rng.integers(-2**50, 2**50, size=n, dtype=np.int64)
    for k in (1, 20, 64, 100, 128):
        check(tk, x, k, item=items, keep=keep)
    for so, ko in ((1, 1), (2, 2), (3, 3), (4, 0), (1, 0), (0, 3)):
        check_views(tk, x, 64, keep, item=items, score_off=so, keep_off=ko)


def test_filter_folded_sparse_and_tail(tk):
    rng = np.random.default_rng(91)
    n = 3_000_017
    x = make("normal", n, 9)
    # So sparse that most first-level rows keep nothing.
    keep = (rng.random(n) < 1e-4).astype(np.uint8)
    for k in (1, 64, 128):
        check(tk, x, k, keep=keep)
    # Kept elements only at the very end (the part after the last full row).
    keep = np.zeros(n, dtype=np.uint8)
    keep[-37:] = 1
    check(tk, x, 64, keep=keep)
    check(tk, x, 20, keep=keep)
    # Only -inf kept, while larger scores are filtered out.
    y = x.copy()
    y[::1000] = -np.inf
    keep = np.zeros(n, dtype=np.uint8)
    keep[::1000] = 1
    check(tk, y, 100, keep=keep)
    # One kept NaN among kept -inf.
    y[5000] = np.nan
    keep[5000] = 1
    check(tk, y, 10, keep=keep)


def test_host_pointers_rejected(tk):
    x = torch.from_numpy(make("normal", 100, 1))
    out_s = torch.empty(5, dtype=torch.float32)
    out_i = torch.empty(5, dtype=torch.int64)
    rc = tk.topk_items_f32_ptr(x.data_ptr(), 0, 0, 100, 5, out_s.data_ptr(), out_i.data_ptr(), 0, 0)
    assert rc == 1


@pytest.mark.parametrize("kind", ["normal", "ties", "specials", "equal"])
def test_large_no_filter_ties_across_rows(tk, kind):
    # From 2^20 positions up the first level cuts the input into ~4096 rows.
    # Ties across rows (every kind but "normal" ties at the k-th score) must
    # still go to the lower position, NaN first and -0 == +0; misaligned
    # bases move the rows' vectors.
    for n, off in ((1 << 20, 0), ((1 << 20) + 4099, 1), (3_000_017, 3)):
        x = make(kind, n, n + 11)
        items = (np.arange(n, dtype=np.int64) * 5 + 1)
        buf = torch.empty(n + off, dtype=torch.float32, device="cuda")
        buf[off:].copy_(torch.from_numpy(x))
        for k in (1, 20, 64, 100, 128):
            s, i, c = tk.topk_items_f32(buf[off:], k, item=torch.from_numpy(items).cuda())
            torch.cuda.synchronize()
            es, ei, ec = oracle.topk_items_f32(x, k, item=items)
            assert int(c.item()) == ec, (kind, n, k)
            assert np.array_equal(i.cpu().numpy(), ei), (kind, n, k)
            assert np.array_equal(bits(s.cpu().numpy()), bits(es)), (kind, n, k)


def test_large_back_to_back(tk):
    # Calls with very different scores, back to back on one stream (each
    # call's scratch is the next one's).
    a = synth.f32_normal(2_000_003, 21) + np.float32(100.0)
    b = synth.f32_normal(1_500_007, 22) - np.float32(100.0)
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    outs = [tk.topk_items_f32(d, 64) for d in (da, db, da, db)]
    torch.cuda.synchronize()
    for (s, i, c), x in zip(outs, (a, b, a, b)):
        es, ei, ec = oracle.topk_items_f32(x, 64)
        assert np.array_equal(i.cpu().numpy(), ei)
        assert np.array_equal(bits(s.cpu().numpy()), bits(es))
