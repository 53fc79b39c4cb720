// CPU oracle for TopK selection -- TEST INFRASTRUCTURE ONLY.
//
// Only the tests, the smoke check and the benchmark's CPU-baseline leg may
// load this library.  The CUDA path never calls it and shares no code with it.
//
// What the pages define ("CUDA parallel optimisation: TopK, shared memory and
// two-stage reduction"):
//   * section 2.1-2.2: gpu_topk(input, output, length, k) keeps the k largest
//     int values; after the second pass the result is stated to be exactly
//     the CPU's result.  The per-thread lists are kept in descending order
//     (section 4.2 shifts smaller entries down), so the output order is
//     descending.
//   * section 6: update_candidates(candidates, k, item, score) -- the same
//     selection keyed by a score that carries an item id: a row of float32
//     scores whose item id is the column index (topk_rows_f32), or one
//     array of scores with item ids and an optional filter in front
//     (topk_items_f32); the section suggests filtering first, then TopK.  The same section
//     names the two-stage reduction pattern as a general tool (sums and
//     other statistics); "CUDA reduction, complete guide" builds it for
//     sums level by level.  oracle_reduce_* are the plain definitions.
//
// The method is exact, so the oracle is the plain definition:
//   topk_i32:      copy, std::sort descending, take the first k.  The output
//                  is the multiset of the k largest values; equal values
//                  appear as often as they occur in the input.
//   topk_rows_f32: per row, std::stable_sort of the column indices by value
//                  descending, take the first k.  Stability makes the lower
//                  column index come first among equal values.
//
// Readings where the pages are silent (each is listed in the design notes):
//   * n == 0, k < 1, k > n, cols < k, rows < 1, null pointers: invalid (-1).
//   * Float order: NaN ranks above +inf and all NaNs are equal to each
//     other; -0.0 and +0.0 are equal (IEEE comparison); +-inf are ordinary.
//     Output values are the input's bits, copied, never recomputed.
//
// Parity pins: every function here is checked by tests that do not reuse it
// (exhaustive brute force on tiny inputs, hand-worked fixtures, closed forms,
// invariants).  The ORACLE_PLANT_* switches exist only so that a test can
// build a deliberately wrong oracle and show that those pins reject it; the
// normal build defines none of them.
#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <functional>
#include <limits>
#include <numeric>
#include <vector>

namespace {

#if defined(ORACLE_PLANT_NAN_LOW)
bool ranks_above(float a, float b) {  // planted mistake: NaN ranked lowest
    bool na = std::isnan(a), nb = std::isnan(b);
    if (na || nb) return !na && nb;
    return a > b;
}
#elif defined(ORACLE_PLANT_SIGNED_ZERO)
bool ranks_above(float a, float b) {  // planted mistake: +0.0 above -0.0
    bool na = std::isnan(a), nb = std::isnan(b);
    if (na || nb) return na && !nb;
    if (a == 0.0f && b == 0.0f) return !std::signbit(a) && std::signbit(b);
    return a > b;
}
#else
// True when a comes strictly before b in the descending score order.
bool ranks_above(float a, float b) {
    bool na = std::isnan(a), nb = std::isnan(b);
    if (na || nb) return na && !nb;
    return a > b;
}
#endif

// IEEE 754 totalOrder, strictly: x comes before y in ascending order.  It
// orders every float bit pattern: -NaN (by payload, larger payloads lower)
// < -inf < ... < -0 < +0 < ... < +inf < +NaN (larger payloads higher).
// It is the order the "GPU radix sort" page's float bit transform gives
// (extensions section: flip every bit of a negative float, only the sign
// bit of a positive one, then compare as unsigned integers); written here
// from the standard's definition, not through that transform.
bool total_less(float x, float y) {
    const bool nx = std::isnan(x), ny = std::isnan(y);
    const bool sx = std::signbit(x), sy = std::signbit(y);
    if (!nx && !ny) {
        if (x < y) return true;
        if (x > y) return false;
        return sx && !sy;  // numerically equal: only -0 < +0 differ
    }
    if (nx && ny) {
        if (sx != sy) return sx;  // -NaN < +NaN
        uint32_t px, py;
        std::memcpy(&px, &x, 4);
        std::memcpy(&py, &y, 4);
        px &= 0x7FFFFFu;
        py &= 0x7FFFFFu;
#if defined(ORACLE_PLANT_NAN_PAYLOAD)
        return px < py;  // planted mistake: negative NaNs ordered like positive ones
#else
        return sx ? px > py : px < py;
#endif
    }
    if (nx) return sx;  // -NaN below every number, +NaN above
    return !sy;         // y is a NaN
}

}  // namespace

extern "C" {

// The k largest of the uint32 values in[0..n) (unsigned order), sorted
// descending, written to out[0..k): the TopK of topk_i32 with unsigned keys.
// Returns 0, or -1 for invalid arguments.
int oracle_topk_u32(const uint32_t* in, size_t n, int k, uint32_t* out) {
    if (!in || !out || n == 0 || k < 1 || (size_t)k > n) return -1;
#if defined(ORACLE_PLANT_U32_SIGNED)
    std::vector<int32_t> v(n);  // planted mistake: compared as signed
    std::memcpy(v.data(), in, n * 4);
    std::sort(v.begin(), v.end(), std::greater<int32_t>());
    std::memcpy(out, v.data(), (size_t)k * 4);
#else
    std::vector<uint32_t> v(in, in + n);
    std::sort(v.begin(), v.end(), std::greater<uint32_t>());
    std::copy(v.begin(), v.begin() + k, out);
#endif
    return 0;
}

// The k largest float32 values of in[0..n) under IEEE 754 totalOrder (see
// total_less), sorted descending, their bits copied to out[0..k).  Every bit
// pattern is its own key, so the output multiset is unique.
// Returns 0, or -1 for invalid arguments.
int oracle_topk_f32(const float* in, size_t n, int k, float* out) {
    if (!in || !out || n == 0 || k < 1 || (size_t)k > n) return -1;
    std::vector<float> v(in, in + n);
#if defined(ORACLE_PLANT_F32_SIGNED_BITS)
    // planted mistake: raw bits compared as signed integers (negatives reversed)
    std::sort(v.begin(), v.end(), [](float a, float b) {
        int32_t x, y;
        std::memcpy(&x, &a, 4);
        std::memcpy(&y, &b, 4);
        return x > y;
    });
#else
    std::sort(v.begin(), v.end(), [](float a, float b) { return total_less(b, a); });
#endif
    std::memcpy(out, v.data(), (size_t)k * 4);
    return 0;
}

// The k largest values of in[0..n), sorted descending, written to out[0..k).
// Returns 0, or -1 for invalid arguments (nothing written).
int oracle_topk_i32(const int32_t* in, size_t n, int k, int32_t* out) {
    if (!in || !out || n == 0 || k < 1 || (size_t)k > n) return -1;
    std::vector<int32_t> v(in, in + n);
#if defined(ORACLE_PLANT_ASCENDING)
    std::sort(v.begin(), v.end());
#else
    std::sort(v.begin(), v.end(), std::greater<int32_t>());
#endif
#if defined(ORACLE_PLANT_DEDUP)
    v.erase(std::unique(v.begin(), v.end()), v.end());  // planted: drops repeats
    if (v.size() < (size_t)k) v.resize((size_t)k, v.back());
#endif
    std::copy(v.begin(), v.begin() + k, out);
    return 0;
}

// Row-wise TopK with indices over a row-major rows x cols float matrix.
// vals and idx are rows x k, row-major: entry j of row r is the j-th best
// (value descending, lower column index first among equal values).
// Returns 0, or -1 for invalid arguments.
int oracle_topk_rows_f32(const float* in, int rows, int cols, int k, float* vals, int32_t* idx) {
    if (!in || !vals || !idx || rows < 1 || cols < 1 || k < 1 || k > cols) return -1;
    std::vector<int32_t> order((size_t)cols);
    for (int r = 0; r < rows; ++r) {
        const float* row = in + (size_t)r * (size_t)cols;
        std::iota(order.begin(), order.end(), 0);
        auto cmp = [row](int32_t a, int32_t b) { return ranks_above(row[a], row[b]); };
#if defined(ORACLE_PLANT_UNSTABLE)
        std::sort(order.begin(), order.end(), cmp);  // planted: tie order lost
#else
        std::stable_sort(order.begin(), order.end(), cmp);
#endif
        for (int j = 0; j < k; ++j) {
            int32_t c = order[(size_t)j];
            idx[(size_t)r * k + j] = c;
            std::memcpy(&vals[(size_t)r * k + j], &row[c], sizeof(float));
        }
    }
    return 0;
}

// Score-keyed TopK with item ids over one array (section 6's
// update_candidates(candidates, k, item, score), composed with a filter as
// the same section suggests): among the positions i with keep[i] != 0 (all
// positions when keep is null), the k best by score in the row order above
// (NaN first, -0 equal to +0, the lower position first among equal scores).
// out_score[j] is the j-th best score (the input's bits), out_item[j] its
// item (item[i], or i when item is null).  When fewer than k positions are
// kept, the rest of the outputs hold -inf and item -1; *out_count is the
// number of real entries.  Returns 0, or -1 for invalid arguments.
int oracle_topk_items_f32(const float* score, const int64_t* item, const uint8_t* keep, size_t n, int k,
                          float* out_score, int64_t* out_item, int64_t* out_count) {
    if (!score || !out_score || !out_item || !out_count || n == 0 || k < 1 || (size_t)k > n) return -1;
    std::vector<int64_t> cand;
    for (size_t i = 0; i < n; ++i)
#if defined(ORACLE_PLANT_KEEP_IGNORED)
        cand.push_back((int64_t)i);  // planted mistake: the filter is ignored
#else
        if (!keep || keep[i]) cand.push_back((int64_t)i);
#endif
    auto cmp = [score](int64_t a, int64_t b) { return ranks_above(score[a], score[b]); };
    std::stable_sort(cand.begin(), cand.end(), cmp);
    const size_t m = cand.size() < (size_t)k ? cand.size() : (size_t)k;
    for (size_t j = 0; j < (size_t)k; ++j) {
        if (j < m) {
            const int64_t i = cand[j];
            std::memcpy(&out_score[j], &score[i], sizeof(float));
            out_item[j] = item ? item[i] : i;
        } else {
            out_score[j] = -std::numeric_limits<float>::infinity();
            out_item[j] = -1;
        }
    }
    *out_count = (int64_t)m;
    return 0;
}

// Radix sort ("GPU radix sort": an LSD radix sort of uint32 keys; its
// extensions section adds key-value pairs).  The result is the keys in
// ascending order, stable: equal keys keep their input order, so each value
// stays with its key and values of equal keys keep their input order.
// vals (and vals_out) may be null for a keys-only sort.  Returns 0, or -1
// for invalid arguments.
int oracle_sort_u32(const uint32_t* keys, const uint32_t* vals, size_t n, uint32_t* keys_out, uint32_t* vals_out) {
    if (!keys || !keys_out || n == 0 || (!vals) != (!vals_out)) return -1;
    std::vector<size_t> order(n);
    std::iota(order.begin(), order.end(), (size_t)0);
#if defined(ORACLE_PLANT_SORT_UNSTABLE)
    std::sort(order.begin(), order.end(), [keys](size_t a, size_t b) { return keys[a] < keys[b]; });  // planted
#else
    std::stable_sort(order.begin(), order.end(), [keys](size_t a, size_t b) { return keys[a] < keys[b]; });
#endif
    for (size_t i = 0; i < n; ++i) {
        keys_out[i] = keys[order[i]];
        if (vals) vals_out[i] = vals[order[i]];
    }
    return 0;
}

// Exact check of a claimed int32 TopK result at any size, in one pass.
//
// out[0..k) is the TopK of in[0..n) exactly when, with t = out[k-1]:
//   out is sorted descending; fewer than k inputs exceed t and at least k
//   inputs are >= t (so t is the k-th largest value); and the inputs greater
//   than t, sorted descending, are exactly out[0..c) with c their count, the
//   rest of out being copies of t.
// Returns 1 if out is the TopK, 0 if not, -1 for invalid arguments.
int oracle_check_topk_i32(const int32_t* in, size_t n, int k, const int32_t* out) {
    if (!in || !out || n == 0 || k < 1 || (size_t)k > n) return -1;
    for (int j = 1; j < k; ++j)
        if (out[j] > out[j - 1]) return 0;
    const int32_t t = out[k - 1];
    std::vector<int32_t> above;
    size_t n_ge = 0;
    for (size_t i = 0; i < n; ++i) {
        if (in[i] >= t) {
            ++n_ge;
            if (in[i] > t) {
                if (above.size() + 1 >= (size_t)k) return 0;  // k or more exceed t
                above.push_back(in[i]);
            }
        }
    }
    if (n_ge < (size_t)k) return 0;
    std::sort(above.begin(), above.end(), std::greater<int32_t>());
    for (size_t j = 0; j < above.size(); ++j)
        if (out[j] != above[j]) return 0;
    for (size_t j = above.size(); j < (size_t)k; ++j)
        if (out[j] != t) return 0;
    return 1;
}

// Reductions (sum, max, min) over int32 and float32 arrays.
//
// op 0 = sum, 1 = max, 2 = min.
//   int32: the sum is exact in int64 (no wrap); max and min are the plain
//          extremes, widened to int64.
//   float32: the sum is accumulated left to right in double (so it differs
//          from the exact sum by at most n * 2^-53 * sum|x|); NaN or
//          +inf + -inf give NaN, as in IEEE arithmetic.  max and min use the
//          IEEE 754-2019 maximum/minimum reading: any NaN gives NaN (written
//          as the canonical quiet NaN), and -0 counts as below +0.  The
//          result is widened to double, which is exact.
// Returns 0, or -1 for invalid arguments.
int oracle_reduce_i32(const int32_t* in, size_t n, int op, int64_t* out) {
    if (!in || !out || n == 0 || op < 0 || op > 2) return -1;
#if defined(ORACLE_PLANT_SUM_WRAP)
    int32_t acc32 = 0;  // planted mistake: a 32-bit accumulator that wraps
    for (size_t i = 0; i < n; ++i) acc32 = (int32_t)((uint32_t)acc32 + (uint32_t)in[i]);
    if (op == 0) {
        *out = acc32;
        return 0;
    }
#endif
    int64_t acc = op == 0 ? 0 : (int64_t)in[0];
    for (size_t i = 0; i < n; ++i) {
        const int64_t x = in[i];
        if (op == 0)
            acc += x;
        else if (op == 1)
            acc = x > acc ? x : acc;
        else
            acc = x < acc ? x : acc;
    }
    *out = acc;
    return 0;
}

int oracle_reduce_f32(const float* in, size_t n, int op, double* out) {
    if (!in || !out || n == 0 || op < 0 || op > 2) return -1;
    if (op == 0) {
        double acc = 0.0;
        for (size_t i = 0; i < n; ++i) acc += (double)in[i];
        *out = acc;
        return 0;
    }
    bool any_nan = false;
    float best = in[0];
    for (size_t i = 0; i < n; ++i) {
        const float x = in[i];
        if (std::isnan(x)) {
            any_nan = true;
            continue;
        }
        if (std::isnan(best)) {
            best = x;
            continue;
        }
#if defined(ORACLE_PLANT_ZERO_ORDER)
        const bool better = op == 1 ? x > best : x < best;  // planted mistake: +-0 ties keep the first
#else
        const bool zeros = x == 0.0f && best == 0.0f;
        const bool better = op == 1 ? (x > best || (zeros && std::signbit(best) && !std::signbit(x)))
                                    : (x < best || (zeros && !std::signbit(best) && std::signbit(x)));
#endif
        if (better) best = x;
    }
    *out = any_nan ? std::numeric_limits<double>::quiet_NaN() : (double)best;
    return 0;
}

}  // extern "C"
