"""Pins for the CPU oracle: it is checked against things other than itself.

* exhaustive brute force on tiny inputs (a different algorithm: repeatedly
  take and remove the best element, written here in plain Python);
* hand-worked fixtures under tests/golden/ (each cites the page section that
  defines the operation);
* closed forms (ascending input, k = 1 is the maximum, k = n is a full
  descending sort done by numpy, all-equal input);
* invariants on random inputs (sorted, sub-multiset, k-th value rank);
* for rows, numpy's stable argsort on inputs without NaN;
* for reductions: Python's exact integers, math.fsum (the correctly rounded
  sum of floats) within the double-precision bound, and an order written
  out with Python keys for max/min over NaN and signed zeros.

The planted-mistake test at the end rebuilds the oracle with one plausible
bug at a time (on the CPU) and shows that at least one pin rejects it.
"""
import collections
import itertools
import math
import struct

import numpy as np
import pytest

import oracle
from _golden import bits, f32_cases, i32_cases, items_cases, reduce_cases, rows_cases, u32_cases

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

INT_MIN, INT_MAX = -(2**31), 2**31 - 1
I32_ALPHABET = [INT_MIN, -1, 0, 1, INT_MAX]
F32_ALPHABET = [math.nan, -math.inf, -1.0, -0.0, 0.0, 1.0, math.inf]


# ---------------------------------------------------------------- helpers --

def brute_topk_i32(values, k):
    """Take the largest remaining value k times."""
    pool = list(values)
    out = []
    for _ in range(k):
        best = max(pool)
        pool.remove(best)
        out.append(best)
    return out


def _rank_key(v):
    # Order used by the brute force below: NaN above everything, then value.
    # -0.0 and +0.0 compare equal under Python float comparison.
    return (1, 0.0) if math.isnan(v) else (0, v)


def brute_topk_row(row, k):
    """Pick the best remaining column k times; the lowest column wins ties."""
    remaining = list(range(len(row)))
    picked = []
    for _ in range(k):
        best = remaining[0]
        for c in remaining[1:]:
            if _rank_key(row[c]) > _rank_key(row[best]):
                best = c
        remaining.remove(best)
        picked.append(best)
    return picked


# Each pin below takes `plant` so the planted-mistake test can rerun it
# against a deliberately wrong oracle build.

def pin_golden_i32(plant=None):
    for x, k, exp in i32_cases():
        got = oracle.topk_i32(x, k, plant=plant)
        assert got.tolist() == exp.tolist(), (x.tolist(), k)


def pin_golden_rows(plant=None):
    for row, k, exp_idx, exp_vals in rows_cases():
        vals, idx = oracle.topk_rows_f32(row[None, :], k, plant=plant)
        assert idx[0].tolist() == exp_idx.tolist(), (row.tolist(), k)
        assert bits(vals[0]).tolist() == bits(exp_vals).tolist(), (row.tolist(), k)


def pin_exhaustive_i32(plant=None, max_n=5):
    for n in range(1, max_n + 1):
        for combo in itertools.product(I32_ALPHABET, repeat=n):
            x = np.array(combo, dtype=np.int32)
            for k in range(1, n + 1):
                got = oracle.topk_i32(x, k, plant=plant).tolist()
                assert got == brute_topk_i32(combo, k), (combo, k)


def pin_exhaustive_rows(plant=None, max_cols=4):
    for cols in range(1, max_cols + 1):
        rows = np.array(list(itertools.product(F32_ALPHABET, repeat=cols)), dtype=np.float32)
        for k in range(1, cols + 1):
            vals, idx = oracle.topk_rows_f32(rows, k, plant=plant)
            for r in range(rows.shape[0]):
                exp = brute_topk_row(rows[r].tolist(), k)
                assert idx[r].tolist() == exp, (rows[r].tolist(), k)
                assert bits(vals[r]).tolist() == bits(rows[r][exp]).tolist()


def pin_closed_forms_i32(plant=None):
    n = 100_003
    asc = np.arange(n, dtype=np.int32)
    for k in (1, 20, 100):
        assert oracle.topk_i32(asc, k, plant=plant).tolist() == list(range(n - 1, n - 1 - k, -1))
    rng = np.random.default_rng(7)
    x = rng.integers(INT_MIN, INT_MAX, size=50_000, endpoint=True, dtype=np.int64).astype(np.int32)
    assert oracle.topk_i32(x, 1, plant=plant)[0] == x.max()
    full = oracle.topk_i32(x, x.size, plant=plant)
    assert np.array_equal(full, np.sort(x)[::-1])
    dup = rng.integers(0, 1000, size=200_000).astype(np.int32)
    assert oracle.topk_i32(dup, 20, plant=plant).tolist() == [999] * 20
    same = np.full(1000, -5, dtype=np.int32)
    assert oracle.topk_i32(same, 999, plant=plant).tolist() == [-5] * 999


def pin_rows_numpy(plant=None):
    # Without NaN the order is numpy's stable argsort of the negated values
    # (-0.0 and +0.0 compare equal in numpy's sort as well).
    rng = np.random.default_rng(11)
    x = np.round(rng.standard_normal((64, 300)) * 4) / 4  # many exact ties
    x = x.astype(np.float32)
    x[0, :5] = [-0.0, 0.0, -0.0, 0.0, 0.0]
    x[1, :] = np.float32(2.0)
    for k in (1, 7, 64, 300):
        vals, idx = oracle.topk_rows_f32(x, k, plant=plant)
        exp_idx = np.argsort(-x, axis=1, kind="stable")[:, :k]
        assert np.array_equal(idx, exp_idx)
        assert np.array_equal(bits(vals), bits(np.take_along_axis(x, exp_idx, axis=1)))


def _same_double(a, b):
    return (math.isnan(a) and math.isnan(b)) or (a == b and math.copysign(1.0, a) == math.copysign(1.0, b))


def pin_golden_reduce(plant=None):
    for dtype, op, x, exp in reduce_cases():
        got = oracle.reduce_i32(x, op, plant=plant) if dtype == "i32" else oracle.reduce_f32(x, op, plant=plant)
        assert got == exp if dtype == "i32" else _same_double(got, exp), (dtype, op, x.tolist(), got, exp)


def _py_extreme(values, op):
    # IEEE 754-2019 maximum/minimum: NaN wins; otherwise order by value, with
    # -0.0 below +0.0 (the sign bit as a tie-break).
    if any(math.isnan(v) for v in values):
        return math.nan
    key = lambda v: (v, math.copysign(1.0, v))
    return max(values, key=key) if op == "max" else min(values, key=key)


def pin_exhaustive_reduce(plant=None, max_n=4):
    for n in range(1, max_n + 1):
        for combo in itertools.product(I32_ALPHABET, repeat=n):
            x = np.array(combo, dtype=np.int32)
            assert oracle.reduce_i32(x, "sum", plant=plant) == sum(combo), combo
            assert oracle.reduce_i32(x, "max", plant=plant) == max(combo), combo
            assert oracle.reduce_i32(x, "min", plant=plant) == min(combo), combo
        for combo in itertools.product(F32_ALPHABET, repeat=min(n, 3)):
            x = np.array(combo, dtype=np.float32)
            vals = [float(v) for v in x]
            for op in ("max", "min"):
                assert _same_double(oracle.reduce_f32(x, op, plant=plant), _py_extreme(vals, op)), (combo, op)
            exact = math.fsum(vals) if not any(math.isnan(v) for v in vals) and not (
                math.inf in vals and -math.inf in vals) else math.nan
            assert _same_double(oracle.reduce_f32(x, "sum", plant=plant) + 0.0, exact + 0.0), combo


def pin_closed_forms_reduce(plant=None):
    n = 100_001
    asc = np.arange(n, dtype=np.int32)
    assert oracle.reduce_i32(asc, "sum", plant=plant) == n * (n - 1) // 2
    big = np.full(70_000, INT_MAX, dtype=np.int32)  # a 32-bit running sum would wrap
    assert oracle.reduce_i32(big, "sum", plant=plant) == 70_000 * INT_MAX
    rng = np.random.default_rng(13)
    x = rng.integers(INT_MIN, INT_MAX, size=200_000, endpoint=True, dtype=np.int64).astype(np.int32)
    assert oracle.reduce_i32(x, "sum", plant=plant) == int(x.astype(np.int64).sum())
    assert oracle.reduce_i32(x, "max", plant=plant) == int(x.max())
    assert oracle.reduce_i32(x, "min", plant=plant) == int(x.min())
    f = (rng.standard_normal(300_000) * 1e3).astype(np.float32)
    s = oracle.reduce_f32(f, "sum", plant=plant)
    vals = f.astype(np.float64)
    bound = f.size * 2.0 ** -53 * float(np.abs(vals).sum())
    assert abs(s - math.fsum(vals.tolist())) <= bound
    assert oracle.reduce_f32(f, "max", plant=plant) == float(f.max())
    assert oracle.reduce_f32(f, "min", plant=plant) == float(f.min())


def pin_golden_items(plant=None):
    for sc, it, kp, k, es, ei, cnt in items_cases():
        s_, i_, c_ = oracle.topk_items_f32(sc, k, item=it, keep=kp, plant=plant)
        assert c_ == cnt and i_.tolist() == ei.tolist(), (sc.tolist(), k, i_.tolist(), c_)
        assert bits(s_).tolist() == bits(es).tolist(), (sc.tolist(), k)


def brute_items(scores, items, keep, k):
    """Pick the best remaining kept position k times (lowest position wins
    ties), then pad."""
    remaining = [i for i in range(len(scores)) if keep is None or keep[i]]
    picked = []
    for _ in range(min(k, len(remaining))):
        best = remaining[0]
        for c in remaining[1:]:
            if _rank_key(scores[c]) > _rank_key(scores[best]):
                best = c
        remaining.remove(best)
        picked.append(best)
    got_items = [items[i] if items is not None else i for i in picked] + [-1] * (k - len(picked))
    return picked, got_items


def pin_exhaustive_items(plant=None, max_n=4):
    for n in range(1, max_n + 1):
        for combo in itertools.product(F32_ALPHABET[:5], repeat=n):
            x = np.array(combo, dtype=np.float32)
            for mask_bits in range(2 ** n):
                keep = np.array([(mask_bits >> i) & 1 for i in range(n)], dtype=np.uint8)
                items = np.arange(100, 100 + n, dtype=np.int64)[::-1].copy()
                for k in range(1, n + 1):
                    s_, i_, c_ = oracle.topk_items_f32(x, k, item=items, keep=keep, plant=plant)
                    picked, exp_items = brute_items(x.tolist(), items.tolist(), keep.tolist(), k)
                    assert c_ == len(picked) and i_.tolist() == exp_items, (combo, keep.tolist(), k)
                    assert bits(s_[:c_]).tolist() == bits(x[picked]).tolist()
                    assert all(math.isinf(v) and v < 0 for v in s_[c_:].tolist())


def pin_items_numpy(plant=None):
    # Without NaN, the kept positions in numpy's stable argsort of the negated
    # scores, first k.
    rng = np.random.default_rng(17)
    x = (np.round(rng.standard_normal(20_000) * 8) / 8).astype(np.float32)  # many ties
    keep = (rng.random(x.size) < 0.3).astype(np.uint8)
    items = rng.integers(-2**62, 2**62, size=x.size, dtype=np.int64)
    kept = np.nonzero(keep)[0]
    order = kept[np.argsort(-x[kept], kind="stable")]
    for k in (1, 50, 1000):
        s_, i_, c_ = oracle.topk_items_f32(x, k, item=items, keep=keep, plant=plant)
        assert c_ == k and i_.tolist() == items[order[:k]].tolist()
        assert bits(s_).tolist() == bits(x[order[:k]]).tolist()
    s_, i_, c_ = oracle.topk_items_f32(x, 64, plant=plant)
    assert i_.tolist() == np.argsort(-x, kind="stable")[:64].tolist()


def pin_golden_sort(plant=None):
    # Hand-worked: "GPU radix sort", sections 2.1 and 8 (key-value pairs):
    # ascending keys, equal keys in input order, values travel with keys.
    keys = np.array([5, 1, 4294967295, 1, 0, 5, 7], dtype=np.uint32)
    vals = np.array([10, 11, 12, 13, 14, 15, 16], dtype=np.uint32)
    ko, vo = oracle.sort_u32(keys, vals, plant=plant)
    assert ko.tolist() == [0, 1, 1, 5, 5, 7, 4294967295]
    assert vo.tolist() == [14, 11, 13, 10, 15, 16, 12]


def pin_exhaustive_sort(plant=None, max_n=5):
    alphabet = [0, 1, 2, 0xFFFFFFFF]
    for n in range(1, max_n + 1):
        for combo in itertools.product(alphabet, repeat=n):
            keys = np.array(combo, dtype=np.uint32)
            vals = np.arange(n, dtype=np.uint32)
            ko, vo = oracle.sort_u32(keys, vals, plant=plant)
            # brute force: take the smallest remaining key, the earliest first
            pool = list(range(n))
            order = []
            while pool:
                best = min(pool, key=lambda i: (combo[i], i))
                pool.remove(best)
                order.append(best)
            assert vo.tolist() == order and ko.tolist() == [combo[i] for i in order], combo


def pin_sort_numpy(plant=None):
    rng = np.random.default_rng(23)
    for n, hi in ((100_000, 2**32), (100_000, 50), (3, 2)):
        keys = rng.integers(0, hi, size=n, dtype=np.uint64).astype(np.uint32)
        vals = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
        order = np.argsort(keys, kind="stable")
        ko, vo = oracle.sort_u32(keys, vals, plant=plant)
        assert np.array_equal(ko, keys[order]) and np.array_equal(vo, vals[order])
        ko2, vo2 = oracle.sort_u32(keys, plant=plant)
        assert np.array_equal(ko2, keys[order]) and vo2 is None


U32_ALPHABET = [0, 1, 2**31 - 1, 2**31, 2**32 - 1]
# Bit patterns: -qNaN payload 1, -qNaN, -inf, -1, -denormal, -0, +0, +denormal, 1, +inf, +qNaN, +qNaN payload 1
F32_PATTERNS = [0xFFC00001, 0xFFC00000, 0xFF800000, 0xBF800000, 0x80000001, 0x80000000, 0x00000000,
                0x00000001, 0x3F800000, 0x7F800000, 0x7FC00000, 0x7FC00001]


def total_order_key(b):
    """IEEE 754 totalOrder as a sort key on a float32 bit pattern, written
    from the standard's description: every non-negative-signed datum above
    every negative-signed one; within a sign, order by magnitude (the
    exponent and significand read as one unsigned number, NaN payloads
    beyond infinity), reversed for the negative sign."""
    mag = b & 0x7FFFFFFF
    return (1, mag) if b >> 31 == 0 else (0, -mag)


def pin_golden_u32(plant=None):
    for x, k, exp in u32_cases():
        assert oracle.topk_u32(x, k, plant=plant).tolist() == exp.tolist(), (x.tolist(), k)


def pin_golden_f32(plant=None):
    for xb, k, expb in f32_cases():
        got = oracle.topk_f32(xb.view(np.float32), k, plant=plant)
        assert bits(got).tolist() == expb.tolist(), ([hex(v) for v in xb], k)


def pin_exhaustive_u32(plant=None, max_n=5):
    for n in range(1, max_n + 1):
        for combo in itertools.product(U32_ALPHABET, repeat=n):
            x = np.array(combo, dtype=np.uint32)
            for k in range(1, n + 1):
                assert oracle.topk_u32(x, k, plant=plant).tolist() == brute_topk_i32(combo, k), (combo, k)


def pin_exhaustive_f32(plant=None, max_n=3):
    for n in range(1, max_n + 1):
        for combo in itertools.product(F32_PATTERNS, repeat=n):
            xb = np.array(combo, dtype=np.uint32)
            exp = sorted(combo, key=total_order_key, reverse=True)
            for k in range(1, n + 1):
                got = bits(oracle.topk_f32(xb.view(np.float32), k, plant=plant)).tolist()
                assert got == exp[:k], ([hex(v) for v in combo], k)


def pin_numpy_u32_f32(plant=None):
    rng = np.random.default_rng(11)
    u = rng.integers(0, 2**32, size=60_000, dtype=np.uint64).astype(np.uint32)
    for k in (1, 7, 1000, u.size):
        assert np.array_equal(oracle.topk_u32(u, k, plant=plant), np.sort(u)[::-1][:k])
    # Numbers only, no zeros and no NaN: totalOrder is numeric order there,
    # so numpy's sort decides.  Magnitudes from denormal to large.
    f = (rng.standard_normal(60_000) * np.exp(rng.uniform(-100, 80, 60_000))).astype(np.float32)
    f = f[f != 0]
    for k in (1, 13, 2000, f.size):
        assert np.array_equal(bits(oracle.topk_f32(f, k, plant=plant)), bits(np.sort(f)[::-1][:k]))
    same = np.full(500, -2.5, dtype=np.float32)
    assert bits(oracle.topk_f32(same, 499, plant=plant)).tolist() == [bits(same)[0]] * 499


ALL_PINS = [pin_golden_u32, pin_golden_f32, pin_exhaustive_u32, pin_exhaustive_f32, pin_numpy_u32_f32,
            pin_golden_i32, pin_golden_rows, pin_exhaustive_i32, pin_exhaustive_rows,
            pin_closed_forms_i32, pin_rows_numpy, pin_golden_reduce, pin_exhaustive_reduce,
            pin_closed_forms_reduce, pin_golden_items, pin_exhaustive_items, pin_items_numpy,
            pin_golden_sort, pin_exhaustive_sort, pin_sort_numpy]


# ------------------------------------------------------------------ tests --

def test_golden_i32():
    pin_golden_i32()


def test_golden_u32_f32():
    pin_golden_u32()
    pin_golden_f32()


def test_exhaustive_u32_f32():
    pin_exhaustive_u32()
    pin_exhaustive_f32()


def test_u32_f32_numpy():
    pin_numpy_u32_f32()


def test_total_order_key_is_numeric_on_numbers():
    # The brute force's key agrees with float comparison on ordered numbers.
    nums = [b for b in F32_PATTERNS if (b & 0x7F800000) != 0x7F800000 or (b & 0x7FFFFF) == 0]
    for a, b in itertools.product(nums, repeat=2):
        fa, fb = struct.unpack("<ff", struct.pack("<II", a, b))
        if fa != fb:
            assert (total_order_key(a) > total_order_key(b)) == (fa > fb), (hex(a), hex(b))


def test_golden_rows():
    pin_golden_rows()


def test_exhaustive_i32_bruteforce():
    pin_exhaustive_i32(max_n=6)


def test_exhaustive_rows_bruteforce():
    pin_exhaustive_rows(max_cols=4)


def test_closed_forms_i32():
    pin_closed_forms_i32()


def test_rows_match_numpy_stable_argsort():
    pin_rows_numpy()


@pytest.mark.parametrize("seed", range(6))
def test_invariants_i32_random(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 20_000))
    k = int(rng.integers(1, n + 1))
    lo, hi = [(INT_MIN, INT_MAX), (-50, 50), (0, 3)][seed % 3]
    x = rng.integers(lo, hi, size=n, endpoint=True, dtype=np.int64).astype(np.int32)
    out = oracle.topk_i32(x, k)
    assert out.size == k
    assert np.all(out[:-1] >= out[1:])
    have = collections.Counter(x.tolist())
    for v, c in collections.Counter(out.tolist()).items():
        assert have[v] >= c
    t = out[-1]
    assert np.count_nonzero(x > t) < k
    assert np.count_nonzero(x >= t) >= k


def test_invariants_rows_random():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((40, 513)).astype(np.float32)
    x[:, ::7] = x[:, :1]  # ties with each row's first value
    k = 33
    vals, idx = oracle.topk_rows_f32(x, k)
    for r in range(x.shape[0]):
        assert len(set(idx[r].tolist())) == k
        assert np.array_equal(bits(vals[r]), bits(x[r, idx[r]]))
        for j in range(1, k):
            a, b = vals[r, j - 1], vals[r, j]
            assert a > b or (a == b and idx[r, j - 1] < idx[r, j])
        kth, kidx = vals[r, -1], idx[r, -1]
        better = np.count_nonzero((x[r] > kth) | ((x[r] == kth) & (np.arange(x.shape[1]) < kidx)))
        assert better == k - 1


def test_nan_payload_bits_are_copied():
    payload = struct.unpack("<f", struct.pack("<I", 0xFFC12345))[0]  # a negative NaN with payload
    row = np.array([1.0, payload, 2.0], dtype=np.float32)
    vals, idx = oracle.topk_rows_f32(row[None, :], 2)
    assert idx[0].tolist() == [1, 2]
    assert bits(vals[0]).tolist() == [0xFFC12345, bits(np.float32(2.0)).item()]


def test_invalid_arguments_rejected():
    x = np.arange(10, dtype=np.int32)
    for k in (0, -1, 11):
        with pytest.raises(oracle.OracleError):
            oracle.topk_i32(x, k)
    with pytest.raises(oracle.OracleError):
        oracle.topk_i32(np.zeros(0, dtype=np.int32), 1)
    m = np.zeros((3, 4), dtype=np.float32)
    for k in (0, 5):
        with pytest.raises(oracle.OracleError):
            oracle.topk_rows_f32(m, k)


# -------------------------------------------------- the exact checker --

def test_checker_accepts_oracle_results():
    rng = np.random.default_rng(5)
    for trial in range(20):
        n = int(rng.integers(1, 5000))
        k = int(rng.integers(1, min(n, 300) + 1))
        x = rng.integers(-40, 40, size=n).astype(np.int32) if trial % 2 else \
            rng.integers(INT_MIN, INT_MAX, size=n, endpoint=True, dtype=np.int64).astype(np.int32)
        assert oracle.check_topk_i32(x, k, oracle.topk_i32(x, k))


def test_checker_rejects_wrong_results():
    x = np.array([5, 3, 3, 9, -1, 3, 7, 7], dtype=np.int32)
    good = oracle.topk_i32(x, 4)  # 9 7 7 5
    assert good.tolist() == [9, 7, 7, 5]
    assert oracle.check_topk_i32(x, 4, good)
    wrong = [
        [9, 7, 7, 3],   # k-th value too small
        [9, 7, 5, 3],   # a repeat dropped
        [9, 9, 7, 7],   # a value repeated more often than in the input
        [7, 9, 7, 5],   # not sorted
        [9, 7, 7, 6],   # 6 is not in the input
        [9, 7, 5, 5],   # 5 occurs once
    ]
    for w in wrong:
        assert not oracle.check_topk_i32(x, 4, np.array(w, dtype=np.int32)), w
    assert not oracle.check_topk_i32(x, 4, good[:3])
    y = np.array([5, 3, 3], dtype=np.int32)
    assert oracle.check_topk_i32(y, 2, np.array([5, 3], dtype=np.int32))
    assert not oracle.check_topk_i32(y, 2, np.array([3, 3], dtype=np.int32))


def test_golden_reduce():
    pin_golden_reduce()


def test_exhaustive_reduce():
    pin_exhaustive_reduce()


def test_closed_forms_reduce():
    pin_closed_forms_reduce()


def test_golden_items():
    pin_golden_items()


def test_exhaustive_items():
    pin_exhaustive_items()


def test_items_numpy():
    pin_items_numpy()


def test_golden_sort():
    pin_golden_sort()


def test_exhaustive_sort():
    pin_exhaustive_sort()


def test_sort_numpy():
    pin_sort_numpy()


def test_reduce_rejects_bad_arguments():
    with pytest.raises(oracle.OracleError):
        oracle.reduce_i32(np.zeros(0, dtype=np.int32), "sum")
    with pytest.raises(KeyError):
        oracle.reduce_f32(np.zeros(3, dtype=np.float32), "mean")


# -------------------------------------------- planted mistakes (CPU only) --

@pytest.mark.parametrize("plant", oracle.PLANTED)
def test_pins_reject_planted_mistake(plant):
    failures = 0
    for pin in ALL_PINS:
        try:
            if pin is pin_exhaustive_i32:
                pin(plant=plant, max_n=4)
            elif pin is pin_exhaustive_rows:
                pin(plant=plant, max_cols=3)
            elif pin is pin_exhaustive_reduce:
                pin(plant=plant, max_n=3)
            elif pin is pin_exhaustive_items:
                pin(plant=plant, max_n=3)
            elif pin is pin_exhaustive_sort:
                pin(plant=plant, max_n=4)
            elif pin is pin_exhaustive_u32:
                pin(plant=plant, max_n=4)
            elif pin is pin_exhaustive_f32:
                pin(plant=plant, max_n=2)
            else:
                pin(plant=plant)
        except AssertionError:
            failures += 1
    assert failures >= 1, f"no pin caught {plant}"
