// Batched float32 row TopK with column indices.
//
// Method: "CUDA parallel optimisation: TopK, shared memory and two-stage
// reduction", section 6 -- update_candidates(candidates, k, item, score):
// the TopK of section 2 keyed by a score that carries an item id.  Here each
// row is one independent selection; the item id is the column.
//
// Order and keys.  A float's bits are mapped to an unsigned key whose integer
// order is the score order ("GPU radix sort", extensions section: floats are
// sorted through a bit transform): negative values have all bits flipped,
// non-negative ones get the sign bit set; -0.0 is first turned into +0.0 so
// the two tie, and every NaN maps to the largest key, above +inf.  The
// 64-bit key (score key << 32) | (0xFFFFFFFF - column) is unique per element
// and its order is "score descending, lower column first", so the selection
// is exact and needs no tie handling beyond comparing keys.
//
// k <= 128: one warp streams each row, keeping its list in registers (see
// the streamed kernel below).  128 < k <= 1024: one block per row with a
// shared-memory candidate buffer.  Output values are decoded from the keys,
// except -0.0 and NaN payloads, which are read again from the row so their
// bits are the input's.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "topk_device.cuh"
#include "topk_internal.h"
#include "topk_sortnet.cuh"

namespace topk {

namespace {


typedef unsigned long long u64;

// Score key: unsigned, order-preserving; -0.0 -> +0.0; NaN -> 0xFFFFFFFF.
__device__ __forceinline__ unsigned score_key(unsigned b) {
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0xFFFFFFFFu;  // NaN
    if (b == 0x80000000u) b = 0u;                               // -0.0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// A float whose score key equals u (used only for the fast compare).
__device__ __forceinline__ float key_float(unsigned u) {
    const unsigned b = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
    return __uint_as_float(b);
}

__device__ __forceinline__ u64 full_key(float v, unsigned col) {
    return ((u64)score_key(__float_as_uint(v)) << 32) | (u64)(0xFFFFFFFFu - col);
}

// max(a, b) that returns NaN when either is NaN (PTX max.NaN).
__device__ __forceinline__ float max_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// ------------------------------------------ k <= 128: streamed rows --
//
// A persistent grid of 3 blocks of 9 warps per SM, so that 4096 rows get one
// warp each on 152 SMs; every warp takes whole rows (rows gw, gw + W, ... for
// global warp gw of W) and needs no other warp.  Each warp owns a ring of
// kRowStages shared-memory stages and keeps bulk copies of its next 3 KiB
// tiles in flight; its tile stream runs on from one row to the next.
// Per row:
//   * start threshold: the k-th largest of 32*GL group maxima of the row's
//     first tile (disjoint groups of real elements, so at least k elements
//     of the row reach it);
//   * every 4-float vector is checked once, by its largest element, against
//     the threshold; flagged vectors are queued as they are, and 32 queued
//     vectors at a time are expanded into exact 64-bit keys, of which those
//     above the threshold are queued again and merged 32 at a time into the
//     warp's sorted register list, whose k-th key raises the threshold;
//   * the warp writes the row's k best (value, column) pairs.
constexpr int kRowWarps = 9;                         // 3 blocks x 9 warps = 27 warps per SM
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kRowU = 6;                             // 16-byte vectors per lane per tile
constexpr int kRowTileVec = 32 * kRowU;              // 3 KiB tiles
constexpr int kRowStages = 2;                        // tiles in flight per warp
constexpr int kRowQueue = 160;                       // per-warp key queue (>= 31 + 4 * 32)
constexpr int kRowVQueue = 48;                       // per-warp vector queue (>= 31 + kRowU)
constexpr int kRowRingBytes = kRowWarps * kRowStages * kRowTileVec * 16;

struct RowGeom {
    const float* rp;
    const float4* body;
    int head, nvec, tail0, ns, tiles;
};

__device__ __forceinline__ RowGeom row_geom(const float* in, int row, int cols) {
    RowGeom g;
    g.rp = in + (size_t)row * (size_t)cols;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(g.rp);
    g.head = (int)(((16u - (unsigned)(addr & 15u)) & 15u) >> 2);
    if (g.head > cols) g.head = cols;
    g.body = reinterpret_cast<const float4*>(g.rp + g.head);
    g.nvec = (cols - g.head) >> 2;
    g.tail0 = g.head + g.nvec * 4;
    g.ns = g.head + (cols - g.tail0);
    g.tiles = (g.nvec + kRowTileVec - 1) / kRowTileVec;
    return g;
}

// Score keys of the largest element of each of a lane's GL groups of kRowU/GL
// float4s (0 for a group with no valid vector; vectors u >= nvalid are not
// valid).
template <int GL>
__device__ __forceinline__ void group_max_keys(const float4 (&r)[kRowU], int nvalid, unsigned (&gk)[GL]) {
#pragma unroll
    for (int j = 0; j < GL; ++j) {
        float fm = -INFINITY;
        bool nan = false, any = false;
#pragma unroll
        for (int u = j * (kRowU / GL); u < (j + 1) * (kRowU / GL); ++u) {
            if (u < nvalid) {
                fm = fmaxf(fmaxf(fm, r[u].x), fmaxf(r[u].y, fmaxf(r[u].z, r[u].w)));
                nan |= (r[u].x != r[u].x) | (r[u].y != r[u].y) | (r[u].z != r[u].z) | (r[u].w != r[u].w);
                any = true;
            }
        }
        gk[j] = !any ? 0u : (nan ? 0xFFFFFFFFu : score_key(__float_as_uint(fm)));
    }
}

// The same over kept elements only: mk[u] holds the keep bytes of vector u
// (byte b for element b; 0 = filtered out).  A group with no kept element
// gives 0.
template <int GL>
__device__ __forceinline__ void group_max_keys_kept(const float4 (&r)[kRowU], const unsigned (&mk)[kRowU],
                                                    int nvalid, unsigned (&gk)[GL]) {
#pragma unroll
    for (int j = 0; j < GL; ++j) {
        float fm = -INFINITY;
        bool nan = false, any = false;
#pragma unroll
        for (int u = j * (kRowU / GL); u < (j + 1) * (kRowU / GL); ++u) {
            if (u < nvalid) {
                const float e[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    if ((mk[u] >> (8 * b)) & 0xFFu) {
                        fm = fmaxf(fm, e[b]);
                        nan |= e[b] != e[b];
                        any = true;
                    }
                }
            }
        }
        gk[j] = !any ? 0u : (nan ? 0xFFFFFFFFu : score_key(__float_as_uint(fm)));
    }
}

// kMask: only elements whose keep byte (same layout as `in`) is nonzero take
// part; each row's outputs hold its valid winners first, then (-inf, -1), and
// row_count[row] says how many are valid.  The keep word of a 16-byte vector
// is read with one 4-byte load (the host checks the alignment that needs).
template <int L, bool kMask>
__global__ void __launch_bounds__(kRowThreads, 3)
topk_rows_stream_kernel(const float* __restrict__ in, int rows, int cols, int k, float* __restrict__ vals,
                        int32_t* __restrict__ idx, unsigned* __restrict__ status, int flags,
                        const uint8_t* __restrict__ keep, int32_t* __restrict__ row_count) {
    constexpr int GL = kRowU;  // groups of 4 elements per lane for the start threshold: 32*GL >= k
    extern __shared__ __align__(128) float4 rring[];       // per-warp stages
    __shared__ __align__(16) u64 s_q[kRowWarps * kRowQueue];  // key queues
    __shared__ __align__(16) float4 s_qv[kRowWarps * kRowVQueue];  // vector queues: values
    __shared__ unsigned s_qc[kRowWarps * kRowVQueue];              // and first columns
    __shared__ __align__(8) uint64_t s_bar[kRowWarps * kRowStages];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRowWarps * kRowStages; ++i) mbar_init(&s_bar[i], 1);
        mbar_init_fence();
    }
    __syncthreads();
    // Launched early (see the host side), this kernel reads only its input
    // until it waits, before its first output write, for the previous
    // kernel on the stream -- or first thing, when that kernel writes its
    // input (kRowsWaitFirst).  It lets the next launch start now when the
    // caller keeps track of what this launch writes (kRowsRelease).
    if (flags & kRowsWaitFirst) grid_dependency_wait();
    if (flags & kRowsRelease) launch_dependents();

    float4* my_ring = rring + (size_t)warp * kRowStages * kRowTileVec;
    uint64_t* my_bar = s_bar + warp * kRowStages;
    u64* q = s_q + warp * kRowQueue;
    float4* qv = s_qv + warp * kRowVQueue;
    unsigned* qc = s_qc + warp * kRowVQueue;
    const int W = gridDim.x * kRowWarps;
    const int gw = blockIdx.x * kRowWarps + warp;

    // Issue side of this warp's tile stream (lane 0): the next (row, tile),
    // with the geometry of that row cached.
    int it_row = gw, it_t = 0;
    RowGeom it_g = row_geom(in, it_row < rows ? it_row : 0, cols);
    size_t issued = 0;
    const uint64_t l2_policy = l2_evict_first_policy();  // the rows are read once
    auto issue_next = [&]() {  // lane 0 only; false when the stream is over
        while (it_row < rows && it_t >= it_g.tiles) {
            it_row += W;
            it_t = 0;
            if (it_row < rows) it_g = row_geom(in, it_row, cols);
        }
        if (it_row >= rows) return false;
        const int base = it_t * kRowTileVec;
        const int cnt = it_g.nvec - base < kRowTileVec ? it_g.nvec - base : kRowTileVec;
        const int st = (int)(issued % kRowStages);
        mbar_arrive_expect_tx(&my_bar[st], (uint32_t)cnt * 16u);
        bulk_copy_g2s_hint(my_ring + (size_t)st * kRowTileVec, it_g.body + base, (uint32_t)cnt * 16u, &my_bar[st],
                           l2_policy);
        ++issued;
        ++it_t;
        return true;
    };
    if (lane == 0)
        for (int i = 0; i < kRowStages; ++i)
            if (!issue_next()) break;
    size_t consumed = 0;
    bool failed = false;

    for (int row = gw; row < rows; row += W) {
        const RowGeom g = row_geom(in, row, cols);
        RegList<L, u64> wl;
        wl.init(0ull);
        u64 T = 0ull;  // only keys above T are kept
        int nq = 0;  // keys in q; below 32 between tiles
        int nv = 0;  // vectors in qv/qc; below 32 between tiles
        // The key queue holds exact keys that beat T when they were queued.
        // A drain takes 32 of them, drops those no longer above T, and merges
        // the rest into the list.
        auto drain = [&](bool all_of_it) {
            while (nq >= 32 || (all_of_it && nq > 0)) {
                const int c = nq >= 32 ? 32 : nq;
                __syncwarp();
                u64 key = lane < c ? q[nq - c + lane] : 0ull;
                __syncwarp();
                nq -= c;
                if (key <= T) key = 0ull;
                const unsigned m = __ballot_sync(kFullMask, key != 0ull);
                if (m) {
                    u64 one[1] = {key};
                    warp_sort_desc<1>(one, lane);
                    wl.merge_sorted32(one[0], __popc(m), lane);
                    if (wl.have >= k) T = kmax(T, warp_sorted_at<L>(wl.lst, k - 1));
                }
            }
        };
        // The exact keys of a vector's elements that beat T; 0 for the
        // others (every real key is above 0).
        auto keys4 = [&](bool has, float4 v, unsigned c0, u64 (&kk)[4]) {
            kk[0] = has ? full_key(v.x, c0 + 0) : 0ull;
            kk[1] = has ? full_key(v.y, c0 + 1) : 0ull;
            kk[2] = has ? full_key(v.z, c0 + 2) : 0ull;
            kk[3] = has ? full_key(v.w, c0 + 3) : 0ull;
            if constexpr (kMask) {
                const unsigned mw =
                    has ? __ldg(reinterpret_cast<const unsigned*>(keep + (size_t)row * (size_t)cols + c0)) : 0u;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (((mw >> (8 * j)) & 0xFFu) == 0u) kk[j] = 0ull;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (kk[j] <= T) kk[j] = 0ull;
        };
        // Queue a lane's (up to 4) nonzero keys with one warp-wide prefix of
        // the counts (0..4, one ballot per bit), then drain full batches.
        // Needs nq < 32 on entry, so that 31 + 4 * 32 fit.
        auto push4 = [&](const u64 (&kk)[4]) {
            const int c = (kk[0] != 0ull) + (kk[1] != 0ull) + (kk[2] != 0ull) + (kk[3] != 0ull);
            const unsigned b0 = __ballot_sync(kFullMask, c & 1), b1 = __ballot_sync(kFullMask, c & 2),
                           b2 = __ballot_sync(kFullMask, c & 4);
            if (c) {
                const unsigned lt = lanemask_lt();
                int o = nq + __popc(b0 & lt) + 2 * __popc(b1 & lt) + 4 * __popc(b2 & lt);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (kk[j]) q[o++] = kk[j];
            }
            nq += __popc(b0) + 2 * __popc(b1) + 4 * __popc(b2);
            if (nq >= 32) drain(false);
        };
        // Expand queued vectors 32 at a time into exact keys and queue those
        // above T (which may have risen since the vectors were flagged).
        auto expand = [&](bool all_of_it) {
            while (nv >= 32 || (all_of_it && nv > 0)) {
                const int c = nv >= 32 ? 32 : nv;
                const bool has = lane < c;
                __syncwarp();
                const float4 v = has ? qv[nv - c + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
                const unsigned c0 = has ? qc[nv - c + lane] : 0u;
                __syncwarp();
                nv -= c;
                u64 kk[4];
                keys4(has, v, c0, kk);
                push4(kk);
            }
        };

        // Scalars outside the aligned body (fewer than 8).
        {
            const int col = lane < g.head ? lane : g.tail0 + (lane - g.head);
            bool has = lane < g.ns;
            if constexpr (kMask) has = has && keep[(size_t)row * (size_t)cols + col] != 0;
            const u64 key = has ? full_key(g.rp[col], (unsigned)col) : 0ull;
            const unsigned m = __ballot_sync(kFullMask, key != 0ull);
            if (key) q[nq + __popc(m & lanemask_lt())] = key;
            nq += __popc(m);
        }

        for (int t = 0; t < g.tiles; ++t) {
            const int stg = (int)(consumed % kRowStages);
            if (!failed && !mbar_wait(&my_bar[stg], (uint32_t)((consumed / kRowStages) & 1))) {
                if (lane == 0) atomicOr(status, kStatusWaitTimeout);
                failed = true;
            }
            const int base = t * kRowTileVec;
            const int cnt = g.nvec - base < kRowTileVec ? g.nvec - base : kRowTileVec;
            const float4* st = my_ring + (size_t)stg * kRowTileVec;
            const int nvalid = cnt > lane ? (cnt - lane + 31) / 32 : 0;  // valid vectors u < nvalid

            if (t == 0) {
                // Start threshold: k-th largest group maximum of the first tile.
                float4 r[kRowU];
#pragma unroll
                for (int u = 0; u < kRowU; ++u)
                    r[u] = u < nvalid ? st[u * 32 + lane] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                unsigned gk[GL];
                if constexpr (kMask) {
                    unsigned mk[kRowU];
                    const uint8_t* krow = keep + (size_t)row * (size_t)cols + g.head;
#pragma unroll
                    for (int u = 0; u < kRowU; ++u)
                        mk[u] = u < nvalid ? __ldg(reinterpret_cast<const unsigned*>(krow + 4 * (u * 32 + lane))) : 0u;
                    group_max_keys_kept<GL>(r, mk, nvalid, gk);
                } else {
                    group_max_keys<GL>(r, nvalid, gk);
                }
                warp_sort_desc<GL>(gk, lane);
                const unsigned seed = warp_sorted_at<GL>(gk, k - 1);
                T = kmax(T, (u64)seed << 32);  // keeps every key with score >= seed
            }

            // Fast pass: which of the lane's vectors hold an element that may
            // beat T (by value, or a tie with a lower column).
            const float tf = key_float((unsigned)(T >> 32));
            const unsigned tc = 0xFFFFFFFFu - (unsigned)T;  // T's column (all columns when T is a bare score)
            unsigned slots = 0u;
#pragma unroll
            for (int u = 0; u < kRowU; ++u) {
                if (u < nvalid) {
                    const float4 v = st[u * 32 + lane];
                    // Largest of the 4, NaN if any is NaN.
                    const float m = max_nan(max_nan(v.x, v.y), max_nan(v.z, v.w));
                    const unsigned c0 = (unsigned)(g.head + (base + u * 32 + lane) * 4);
                    if (!(m <= tf) || (m == tf && c0 < tc)) slots |= 1u << u;
                }
            }
            // Slow pass: the flagged vectors go to the vector queue as they
            // are, placed with one warp-wide prefix of the per-lane counts
            // (0..kRowU, one ballot per bit); expand() turns them into keys.
            if (__any_sync(kFullMask, slots != 0u)) {
                static_assert(kRowU < 8, "three ballots count 0..7 vectors");
                const int c = __popc(slots);
                const unsigned lt = lanemask_lt();
                int off = 0, total = 0;
#pragma unroll
                for (int bit = 0; bit < 3; ++bit) {
                    const unsigned bb = __ballot_sync(kFullMask, (c >> bit) & 1);
                    off += __popc(bb & lt) << bit;
                    total += __popc(bb) << bit;
                }
                if (nv + total > kRowVQueue) expand(true);
                if (total <= kRowVQueue) {
                    int o = nv + off;
#pragma unroll
                    for (int u = 0; u < kRowU; ++u) {
                        if ((slots >> u) & 1u) {
                            qv[o] = st[u * 32 + lane];
                            qc[o] = (unsigned)(g.head + (base + u * 32 + lane) * 4);
                            ++o;
                        }
                    }
                    nv += total;
                    if (nv >= 32) expand(false);
                } else {
                    // More flagged vectors than the queue holds (a weak
                    // threshold early in a row): one vector position at a
                    // time, straight to keys.
                    unsigned todo = __reduce_or_sync(kFullMask, slots);
#pragma unroll 1
                    while (todo) {
                        const int u = __ffs(todo) - 1;
                        todo &= todo - 1;
                        const bool has = (slots >> u) & 1u;
                        const float4 v = has ? st[u * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
                        u64 kk[4];
                        keys4(has, v, (unsigned)(g.head + (base + u * 32 + lane) * 4), kk);
                        push4(kk);
                    }
                }
            }
            __syncwarp();
            ++consumed;
            if (lane == 0 && !failed) {
                fence_proxy_async_smem();
                issue_next();
            }
        }
        expand(true);
        drain(true);

        // The row's k best.  The key gives the value back exactly except for
        // -0.0 (keyed as +0.0) and NaN payloads: those are read from the row.
        grid_dependency_wait();  // the previous kernel's writes come first
        int valid = 0;
#pragma unroll
        for (int j = 0; j < L; ++j) {
            const int p = j * 32 + lane;
            if constexpr (kMask) valid += __popc(__ballot_sync(kFullMask, p < k && wl.lst[j] != 0ull));
            if (p < k) {
                const u64 key = wl.lst[j];
                const unsigned col = 0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull);
                const unsigned u = (unsigned)(key >> 32);
                float v;
                if (kMask && key == 0ull) {
                    v = __int_as_float(0xFF800000);  // fewer than k kept elements: (-inf, -1)
                    vals[(size_t)row * k + p] = v;
                    idx[(size_t)row * k + p] = -1;
                    continue;
                }
                if (col >= (unsigned)cols)
                    v = __int_as_float(0x7fc00000);  // unreachable: every list entry is a real element
                else if (u == 0x80000000u || u == 0xFFFFFFFFu)
                    v = g.rp[col];
                else
                    v = key_float(u);
                vals[(size_t)row * k + p] = v;
                idx[(size_t)row * k + p] = (int32_t)col;
            }
        }
        if constexpr (kMask)
            if (lane == 0) row_count[row] = valid;
    }
    // After a wait gave up, let the copies still in flight land before exit.
    if (lane == 0)
        for (size_t c = consumed; c < issued; ++c)
            if (!mbar_wait(&my_bar[c % kRowStages], (uint32_t)((c / kRowStages) & 1))) break;
}

// ------------------------------------- 128 < k <= 1024: one block per row --
//
// Each block streams its rows (rows b, b + G, ... for block b of G) through
// a ring of kBigStages shared-memory stages of 8 KiB, filled by bulk copies
// that thread 0 keeps in flight across row boundaries.  A round consumes one
// stage: every thread checks one 16-byte vector, by its largest element,
// against the block's threshold T (a lower bound of the row's k-th key);
// flagged vectors go to the warp's queue, and once 32 are queued the warp
// expands them into exact 64-bit keys, of which those above T go to a shared
// candidate buffer (one atomic per warp).  So most rounds cost a warp a
// compare and a ballot, however many of its warps' vectors pass.  T only
// rises and stays below the row's k-th key, so every key of the row's k best
// reaches the buffer and stays there.
//
// Cutting the buffer is a radix select, not a sort.  Its keys share a
// common prefix (found with one OR-reduction of key ^ buf[0]); histograms of
// the next 11 bits narrow down the bucket that holds the k-th largest key
// until the keys at or above that bucket's lower edge L number at most
// `limit`.  Those keys stay, and T becomes L - 1.  At the row's end a cut
// with limit k leaves exactly the k best keys, which a bitonic sort orders.
constexpr int kBigThreads = 512;
constexpr int kBigStageVec = kBigThreads;    // 16-byte vectors per stage (one per thread)
constexpr int kBigStages = 6;                // stages in flight per block (48 KiB)
constexpr int kBigCap = 4096;                // candidate buffer (32 KiB)
constexpr int kBigRound = kBigStageVec * 4;  // keys one round can add
constexpr int kBigKeep = kBigCap - kBigRound;  // most keys a cut may keep
constexpr int kBigDigit = 11;
constexpr int kBigBins = 1 << kBigDigit;
constexpr int kBigPer = kBigCap / kBigThreads;  // buffer keys per thread
constexpr int kBigSlack = 256;                 // keys above k that a cut inside the row may keep
constexpr int kBigQueue = 64;                  // per-warp vector queue (>= 31 + 32)
constexpr int kBigRingBytes = kBigStages * kBigStageVec * 16;
static_assert(1024 + kBigSlack <= kBigKeep, "k <= 1024 best keys plus the slack fit");
static_assert(kBigBins == 4 * kBigThreads, "the bin scan gives each thread four bins");
static_assert(kBigRound >= (kBigThreads / 32) * 32 * 4, "a round's queue drains add at most kBigRound keys");

// Append a thread's keys (those that are nonzero) to buf at *cnt: a
// warp-wide prefix of the per-thread counts (one ballot per bit of the
// count) and one shared atomic per warp.  Returns the warp's end position in
// the buffer (the largest such end is the buffer's count).  Keys past
// kBigCap are dropped (the callers' cuts keep the buffer below it; this only
// bounds the writes).
template <int N>
__device__ __forceinline__ unsigned big_append(const u64 (&kk)[N], u64* buf, unsigned* cnt, int lane) {
    constexpr int kBits = N < 2 ? 1 : (N < 4 ? 2 : (N < 8 ? 3 : 4));
    int c = 0;
#pragma unroll
    for (int j = 0; j < N; ++j) c += kk[j] != 0ull;
    const unsigned lt = lanemask_lt();
    int tot = 0, before = 0;
#pragma unroll
    for (int b = 0; b < kBits; ++b) {
        const unsigned m = __ballot_sync(kFullMask, (c >> b) & 1);
        tot += __popc(m) << b;
        before += __popc(m & lt) << b;
    }
    unsigned base = 0;
    if (lane == 0 && tot) base = atomicAdd(cnt, (unsigned)tot);
    base = __shfl_sync(kFullMask, base, 0);
    int o = (int)base + before;
#pragma unroll
    for (int j = 0; j < N; ++j)
        if (kk[j]) {
            if (o < kBigCap) buf[o] = kk[j];
            ++o;
        }
    return tot ? base + (unsigned)tot : 0u;
}

__global__ void __launch_bounds__(kBigThreads, 2)
topk_rows_big_kernel(const float* __restrict__ in, int rows, int cols, int k, float* __restrict__ vals,
                     int32_t* __restrict__ idx, unsigned* __restrict__ status) {
    extern __shared__ __align__(128) float4 bring[];  // kBigStages stages
    __shared__ __align__(16) u64 buf[kBigCap];
    __shared__ __align__(16) unsigned hist[kBigBins];
    __shared__ __align__(16) float4 s_qv[(kBigThreads / 32) * kBigQueue];  // queued vectors
    __shared__ unsigned s_qi[(kBigThreads / 32) * kBigQueue];               // and their vector index
    __shared__ __align__(8) uint64_t s_bar[kBigStages];
    __shared__ unsigned s_wsum[kBigThreads / 32];
    __shared__ unsigned s_or[2];
    __shared__ unsigned s_cnt, s_bin, s_above, s_inbin, s_fail;
    __shared__ u64 s_T;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int i = 0; i < kBigStages; ++i) mbar_init(&s_bar[i], 1);
        mbar_init_fence();
        s_or[0] = s_or[1] = 0u;
        s_fail = 0u;
    }
    __syncthreads();

    // Issue side (thread 0): the next (row, tile) of this block's stream,
    // with that row's geometry.  refill(released) keeps tiles up to
    // released + kBigStages - 1 in flight, where the first `released`
    // consumed tiles are those whose reads a block barrier has followed.
    // The issue state lives in shared memory: only thread 0 uses it.
    __shared__ const float4* s_it_body;
    __shared__ int s_it_row, s_it_base, s_it_nvec;
    __shared__ unsigned s_issued;
    unsigned consumed = 0;
    const uint64_t l2_policy = l2_evict_first_policy();  // the rows are read once
    auto refill = [&](unsigned released) {  // thread 0
        int it_row = s_it_row, it_base = s_it_base, it_nvec = s_it_nvec;
        const float4* it_body = s_it_body;
        unsigned issued = s_issued;
        while (issued < released + kBigStages) {
            while (it_row < rows && it_base >= it_nvec) {
                it_row += gridDim.x;
                it_base = 0;
                if (it_row < rows) {
                    const RowGeom ig = row_geom(in, it_row, cols);
                    it_body = ig.body;
                    it_nvec = ig.nvec;
                }
            }
            if (it_row >= rows) break;
            const int n = it_nvec - it_base < kBigStageVec ? it_nvec - it_base : kBigStageVec;
            const int st = (int)(issued % kBigStages);
            mbar_arrive_expect_tx(&s_bar[st], (uint32_t)n * 16u);
            bulk_copy_g2s_hint(bring + (size_t)st * kBigStageVec, it_body + it_base, (uint32_t)n * 16u, &s_bar[st],
                               l2_policy);
            ++issued;
            it_base += kBigStageVec;
        }
        s_it_row = it_row;
        s_it_base = it_base;
        s_it_nvec = it_nvec;
        s_it_body = it_body;
        s_issued = issued;
    };
    if (tid == 0) {
        const RowGeom g0 = row_geom(in, blockIdx.x < rows ? blockIdx.x : 0, cols);
        s_it_row = blockIdx.x;
        s_it_base = 0;
        s_it_nvec = (int)blockIdx.x < rows ? g0.nvec : 0;
        s_it_body = g0.body;
        s_issued = 0u;
        refill(0u);
    }

    // Cut the buffer (every thread, after a barrier; s_cnt >= k): keep the
    // keys at or above the lower edge L of the smallest bucket that holds
    // the k-th largest key and has at most `limit` keys at or above it;
    // T = L - 1.
    auto cut = [&](unsigned limit) {
        const unsigned cnt = kmin(s_cnt, (unsigned)kBigCap);
        const int nj = (int)((cnt + kBigThreads - 1) / kBigThreads);  // key slots in use (block-uniform)
        u64 kv[kBigPer];
#pragma unroll
        for (int j = 0; j < kBigPer; ++j) {
            const unsigned i = (unsigned)(tid + j * kBigThreads);
            kv[j] = j < nj && i < cnt ? buf[i] : 0ull;  // real keys are nonzero
        }
        const u64 x0 = buf[0];
        u64 d = 0ull;
#pragma unroll
        for (int j = 0; j < kBigPer; ++j)
            if (kv[j]) d |= kv[j] ^ x0;
        const unsigned dh = __reduce_or_sync(kFullMask, (unsigned)(d >> 32));
        const unsigned dl = __reduce_or_sync(kFullMask, (unsigned)d);
        if (lane == 0) {
            if (dh) atomicOr(&s_or[0], dh);
            if (dl) atomicOr(&s_or[1], dl);
        }
        __syncthreads();
        const u64 dall = ((u64)s_or[0] << 32) | (u64)s_or[1];
        if (tid == 0) s_cnt = 0u;  // every thread has read it
        int pb = dall ? __clzll((long long)dall) : 64;  // bits every key shares
        u64 P = pb == 0 ? 0ull : (pb == 64 ? x0 : x0 >> (64 - pb));
        unsigned above = 0u;  // keys above the current bucket
        u64 L = x0;
        while (pb < 64) {
            const int D = 64 - pb < kBigDigit ? 64 - pb : kBigDigit;
            const int shift = 64 - pb - D;
            reinterpret_cast<uint4*>(hist)[tid] = make_uint4(0u, 0u, 0u, 0u);
            const u64 hmask = pb == 0 ? 0ull : ~0ull << (64 - pb);  // the bucket's known bits
            const u64 hval = pb == 0 ? 0ull : P << (64 - pb);
            __syncthreads();
#pragma unroll
            for (int j = 0; j < kBigPer; ++j)
                if (j < nj && kv[j] && (kv[j] & hmask) == hval)
                    atomicAdd(&hist[(unsigned)(kv[j] >> shift) & (kBigBins - 1)], 1u);
            __syncthreads();
            // Thread t takes bins 4t'..4t'+3 with t' = kBigThreads-1-t, so the
            // threads run from the top bin down.
            const uint4 h4 = reinterpret_cast<const uint4*>(hist)[kBigThreads - 1 - tid];
            const unsigned hq[4] = {h4.w, h4.z, h4.y, h4.x};
            const unsigned s = hq[0] + hq[1] + hq[2] + hq[3];
            unsigned incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(kFullMask, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) s_wsum[warp] = incl;
            __syncthreads();
            unsigned c = above + incl - s;
            for (int w = 0; w < warp; ++w) c += s_wsum[w];
            if (c < (unsigned)k && c + s >= (unsigned)k) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (c < (unsigned)k && c + hq[q] >= (unsigned)k) {
                        s_bin = (unsigned)(4 * (kBigThreads - 1 - tid) + 3 - q);
                        s_above = c;
                        s_inbin = hq[q];
                    }
                    c += hq[q];
                }
            }
            __syncthreads();
            const unsigned b = s_bin;
            above = s_above;
            const unsigned inb = s_inbin;
            P = (P << D) | (u64)b;
            pb += D;
            L = shift ? P << shift : P;
            if (above + inb <= limit) break;
            __syncthreads();  // s_wsum, s_bin, hist are rewritten by the next pass
        }
#pragma unroll
        for (int j = 0; j < kBigPer; ++j)
            if (!(j < nj && kv[j] >= L)) kv[j] = 0ull;
        big_append<kBigPer>(kv, buf, &s_cnt, lane);
        if (tid == 0) {
            s_T = L ? L - 1 : 0ull;
            s_or[0] = s_or[1] = 0u;
        }
        __syncthreads();
    };

    float4* qv = s_qv + warp * kBigQueue;
    unsigned* qi = s_qi + warp * kBigQueue;
    for (int row = blockIdx.x; row < rows; row += gridDim.x) {
        const RowGeom g = row_geom(in, row, cols);
        int nq = 0;  // vectors in this warp's queue (warp-uniform); below 32 between rounds
        // The end of this warp's last append since the last barrier.  A
        // barrier that ORs (hi > kBigKeep) tells every thread, alike, whether
        // the buffer holds more than kBigKeep keys -- reading the count
        // instead would race with warps that have already moved on and
        // append.
        unsigned hi = 0u;
        // Expand the warp's last c <= 32 queued vectors into keys above T and
        // append them to the buffer.
        auto drain = [&](int c, u64 T) {
            __syncwarp();
            u64 kk[4] = {0ull, 0ull, 0ull, 0ull};
            if (lane < c) {
                const float4 v = qv[nq - c + lane];
                const unsigned c0 = (unsigned)g.head + 4u * qi[nq - c + lane];
                const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const u64 key = full_key(e[j], c0 + j);
                    kk[j] = key > T ? key : 0ull;
                }
            }
            __syncwarp();  // read before the slots are queued to again
            nq -= c;
            hi = kmax(hi, big_append<4>(kk, buf, &s_cnt, lane));
        };
        if (tid == 0) {
            s_cnt = 0u;
            s_T = 0ull;
        }
        __syncthreads();
        // Scalars outside the aligned body (fewer than 8): warp 0.
        if (tid < 32) {
            const int col = lane < g.head ? lane : g.tail0 + (lane - g.head);
            const u64 kk[1] = {lane < g.ns ? full_key(g.rp[col], (unsigned)col) : 0ull};
            hi = big_append<1>(kk, buf, &s_cnt, lane);
        }
        const int tiles = (g.nvec + kBigStageVec - 1) / kBigStageVec;
        for (int t = 0; t < tiles; ++t) {
            // Thread 0 alone waits for this round's stage; the barrier hands
            // the landed data to the block (and the other threads sleep
            // there instead of polling).
            const int st = (int)(consumed % kBigStages);
            if (tid == 0 && !mbar_wait(&s_bar[st], (uint32_t)((consumed / kBigStages) & 1))) {
                atomicOr(status, kStatusWaitTimeout);
                s_fail = 1u;
            }
            // The last round's keys are in, its stage is read, this one has landed.
            const bool full = __syncthreads_or(hi > (unsigned)kBigKeep);
            hi = 0u;
            if (s_fail) break;
            const unsigned released = consumed;
            ++consumed;
            if (full) cut((unsigned)k + kBigSlack);
            const u64 T = s_T;
            const float tf = key_float((unsigned)(T >> 32));
            const int i = t * kBigStageVec + tid;
            // A vector whose largest element (NaN if it holds one) is not
            // below T's score may hold a key above T: queue it.
            bool flag = false;
            float4 v;
            if (i < g.nvec) {
                v = bring[(size_t)st * kBigStageVec + tid];
                flag = !(max_nan(max_nan(v.x, v.y), max_nan(v.z, v.w)) < tf);
            }
            const unsigned bal = __ballot_sync(kFullMask, flag);
            if (bal) {
                if (flag) {
                    const int pos = nq + __popc(bal & lanemask_lt());
                    qv[pos] = v;
                    qi[pos] = (unsigned)i;
                }
                nq += __popc(bal);
                if (nq >= 32) drain(32, T);
            }
            if (tid == 0) refill(released);
        }
        const bool full = __syncthreads_or(hi > (unsigned)kBigKeep);
        if (s_fail) break;
        if (tid == 0) refill(consumed);
        // Empty the queues (at most 31 vectors each, after a cut if the
        // buffer could not take them), then a cut with limit k leaves the k
        // best keys.  (No warp appends between a barrier and the next cut's
        // first barrier, so the cut and the test below read a settled count.)
        if (full) cut((unsigned)k + kBigSlack);
        if (nq) drain(nq, s_T);
        __syncthreads();
        if (s_cnt >= (unsigned)k) cut((unsigned)k);
        const int n = (int)kmin(s_cnt, (unsigned)kBigCap);  // k (fewer only if the row were shorter than k)
        const int L2 = next_pow2(n < 64 ? 64 : n);
        for (int j = n + tid; j < L2; j += kBigThreads) buf[j] = 0ull;  // below every real key
        if (L2 <= 2 * kBigThreads)
            block_sort_reg_desc<u64, kBigThreads>(buf, L2);
        else
            block_sort_smem_desc(buf, L2);
        for (int j = tid; j < k; j += kBigThreads) {
            const u64 key = j < n ? buf[j] : 0ull;
            const unsigned col = 0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull);
            const unsigned u = (unsigned)(key >> 32);
            float v;
            if (col >= (unsigned)cols)
                v = __int_as_float(0x7fc00000);  // unreachable: the row has at least k elements
            else if (u == 0x80000000u || u == 0xFFFFFFFFu)
                v = g.rp[col];  // -0.0 and NaN payloads: the input's bits
            else
                v = key_float(u);
            vals[(size_t)row * k + j] = v;
            idx[(size_t)row * k + j] = (int32_t)col;
        }
        __syncthreads();  // the buffer is reused by the next row
    }
    // After a wait gave up, let the copies still in flight land before exit.
    if (tid == 0)
        for (unsigned c = consumed; c < s_issued; ++c)
            if (!mbar_wait(&s_bar[c % kBigStages], (uint32_t)((c / kBigStages) & 1))) break;
}

// ------------------------------- 128 < k <= 1024, rows up to 64K columns --
//
// One block per row at a time (a persistent grid; block b takes rows b,
// b + G, ...): a radix select on the row's unique 64-bit keys (score key,
// inverted column), as in "GPU radix sort"'s histogram section, 11-bit
// digits:
//   * a pass over the row histograms the next digit of the keys that share
//     the bits fixed so far (the first pass reads the row from HBM, the
//     later ones find it in L2);
//   * the bucket that holds the need-th largest key is picked; when all the
//     keys at or above that bucket's lower edge fit the candidate buffer, a
//     last pass collects them, else the bucket's digit is fixed and the next
//     digit is histogrammed.  The keys are unique, so the last level's
//     bucket holds one key and the buffer always suffices by then;
//   * when the candidates round to the same sort size as k they are all
//     sorted; else the select goes on over them in shared memory until
//     exactly the k best are left, and those are sorted; the first k are
//     written.
// For N(0,1) rows and k = 129 .. 1024 one level is enough (about 200 .. 1300
// candidates), so a row is read once from HBM and once from L2.  Four
// 256-thread blocks per SM keep that many rows in flight.
constexpr int kSelThreads = 256;
constexpr int kSelCap = 4096;                 // candidate buffer (32 KiB)
constexpr int kSelBits = 11;
constexpr int kSelBins = 1 << kSelBits;
constexpr int kSelU = 8;                      // 16-byte loads in flight per thread
constexpr int kSelPer = kSelBins / kSelThreads;  // bins per thread in the bucket scan
static_assert(kSelPer * kSelThreads == kSelBins, "the bucket scan covers the bins");
static_assert(1024 <= kSelCap, "k <= 1024");
static_assert(kSelBins * sizeof(unsigned) >= 1024 * sizeof(u64), "the histogram's space holds the k <= 1024 best");


__global__ void __launch_bounds__(kSelThreads, 4)
topk_rows_select_kernel(const float* __restrict__ in, int rows, int cols, int k, float* __restrict__ vals,
                        int32_t* __restrict__ idx) {
    __shared__ __align__(16) u64 buf[kSelCap];
    __shared__ __align__(16) unsigned hist[kSelBins];
    __shared__ unsigned s_wsum[kSelThreads / 32];
    __shared__ unsigned s_digit, s_above, s_cnt, s_n;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int row = blockIdx.x; row < rows; row += gridDim.x) {
        const RowGeom g = row_geom(in, row, cols);
        // f(v, col, ok) for every element of the row, warp-uniform calls:
        // the 16-byte body in batches of kSelU loads per thread, then the
        // few scalars outside it in warp 0.
        auto for_row = [&](auto f) {
            for (int base = 0; base < g.nvec; base += kSelThreads * kSelU) {
                float4 r[kSelU];
#pragma unroll
                for (int u = 0; u < kSelU; ++u) {
                    const int i = base + u * kSelThreads + tid;
                    r[u] = i < g.nvec ? g.body[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kSelU; ++u) {
                    const int i = base + u * kSelThreads + tid;
                    const bool ok = i < g.nvec;
                    const unsigned c = (unsigned)(g.head + 4 * i);
                    f(r[u].x, c, ok);
                    f(r[u].y, c + 1u, ok);
                    f(r[u].z, c + 2u, ok);
                    f(r[u].w, c + 3u, ok);
                }
            }
            if (warp == 0) {
                const bool ok = lane < g.ns;
                const int c = lane < g.head ? lane : g.tail0 + (lane - g.head);
                f(ok ? g.rp[c] : 0.f, (unsigned)c, ok);
            }
        };

        // The bucket of hist (complete after a barrier) that holds the
        // want-th largest counted key: s_digit, with s_above keys in higher
        // buckets and s_cnt in it.  Thread t takes bins 2047 - kSelPer t - q.
        auto pick = [&](unsigned want) {
            unsigned c[kSelPer], sum = 0;
#pragma unroll
            for (int q = 0; q < kSelPer; ++q) {
                c[q] = hist[kSelBins - 1 - kSelPer * tid - q];
                sum += c[q];
            }
            unsigned x = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(kFullMask, x, o);
                if (lane >= o) x += y;
            }
            if (lane == 31) s_wsum[warp] = x;
            __syncthreads();
            unsigned acc = x - sum;
            for (int w = 0; w < warp; ++w) acc += s_wsum[w];
#pragma unroll
            for (int q = 0; q < kSelPer; ++q) {
                if (acc < want && want <= acc + c[q]) {
                    s_digit = (unsigned)(kSelBins - 1 - kSelPer * tid - q);
                    s_above = acc;
                    s_cnt = c[q];
                }
                acc += c[q];
            }
            __syncthreads();
        };

        // Select: fix 11-bit digits from the top until the keys at or above
        // the chosen bucket fit the buffer.
        u64 prefix = 0ull;  // the fixed bits [top, 64)
        int top = 64;
        unsigned need = (unsigned)k;
        for (;;) {
            const int shift = top > kSelBits ? top - kSelBits : 0;
            const unsigned dmask = (1u << (top - shift)) - 1u;
            for (int i = tid; i < kSelBins; i += kSelThreads) hist[i] = 0u;
            __syncthreads();
            if (top == 64) {
                for_row([&](float v, unsigned, bool ok) {
                    if (ok) atomicAdd(&hist[score_key(__float_as_uint(v)) >> (32 - kSelBits)], 1u);
                });
            } else {
                const u64 fixed = prefix >> top;
                for_row([&](float v, unsigned c, bool ok) {
                    const u64 key = full_key(v, c);
                    if (ok && (key >> top) == fixed) atomicAdd(&hist[(unsigned)(key >> shift) & dmask], 1u);
                });
            }
            __syncthreads();
            pick(need);
            const unsigned total = ((unsigned)k - need) + s_above + s_cnt;  // keys at or above the bucket
            prefix |= (u64)s_digit << shift;
            need -= s_above;
            // All of the bucket is needed: the keys at or above its lower
            // edge are the k best (top = 0 marks that).
            top = need == s_cnt ? 0 : shift;
            if (total <= (unsigned)kSelCap || top == 0) break;
        }

        // Collect the keys at or above prefix (its bits below `top` are zero):
        // a float compare of each vector's largest element against the
        // bucket's score first (every element at or above it passes, NaN
        // included); keys only for vectors that pass, and one shared-counter
        // add per warp and vector round that has any.
        if (tid == 0) s_n = 0u;
        __syncthreads();
        {
            const float tf = key_float((unsigned)(prefix >> 32));
            // Append this lane's keys of one round (m: which of the 4 pass).
            auto append = [&](unsigned m, u64 k0, u64 k1, u64 k2, u64 k3) {
                const unsigned cnt = __popc(m);
                unsigned x = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(kFullMask, x, o);
                    if (lane >= o) x += y;
                }
                unsigned at = 0;
                if (lane == 31 && x) at = atomicAdd(&s_n, x);
                at = __shfl_sync(kFullMask, at, 31) + (x - cnt);
                if ((m & 1u) && at < (unsigned)kSelCap) buf[at] = k0;
                at += m & 1u;
                if ((m & 2u) && at < (unsigned)kSelCap) buf[at] = k1;
                at += (m >> 1) & 1u;
                if ((m & 4u) && at < (unsigned)kSelCap) buf[at] = k2;
                at += (m >> 2) & 1u;
                if ((m & 8u) && at < (unsigned)kSelCap) buf[at] = k3;
            };
            for (int base = 0; base < g.nvec; base += kSelThreads * kSelU) {
                float4 r[kSelU];
#pragma unroll
                for (int u = 0; u < kSelU; ++u) {
                    const int i = base + u * kSelThreads + tid;
                    r[u] = i < g.nvec ? g.body[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kSelU; ++u) {
                    const int i = base + u * kSelThreads + tid;
                    const bool pass = i < g.nvec && !(max_nan(max_nan(r[u].x, r[u].y), max_nan(r[u].z, r[u].w)) < tf);
                    if (__any_sync(kFullMask, pass)) {
                        const unsigned c = (unsigned)(g.head + 4 * i);
                        const u64 k0 = full_key(r[u].x, c), k1 = full_key(r[u].y, c + 1u);
                        const u64 k2 = full_key(r[u].z, c + 2u), k3 = full_key(r[u].w, c + 3u);
                        const unsigned m = pass ? (k0 >= prefix ? 1u : 0u) | (k1 >= prefix ? 2u : 0u) |
                                                      (k2 >= prefix ? 4u : 0u) | (k3 >= prefix ? 8u : 0u)
                                                : 0u;
                        append(m, k0, k1, k2, k3);
                    }
                }
            }
            if (warp == 0) {
                const bool ok = lane < g.ns;
                const int c = lane < g.head ? lane : g.tail0 + (lane - g.head);
                const u64 key = full_key(ok ? g.rp[c] : 0.f, (unsigned)c);
                append(ok && key >= prefix ? 1u : 0u, key, 0ull, 0ull, 0ull);
            }
        }
        __syncthreads();
        const int n = (int)kmin(s_n, (unsigned)kSelCap);  // >= k

        // The k best of the candidates.  When they round to the same sort
        // size as k, sort them all.  Else go on with the select in shared
        // memory (the keys are unique) until the keys at or above prefix are
        // exactly the k best, move those to `best` (the histogram's space)
        // and sort them.
        u64* best = buf;
        int nb = n;
        if (top > 0 && next_pow2(n < 64 ? 64 : n) > next_pow2(k < 64 ? 64 : k)) {
            while (top > 0) {
                const int shift = top > kSelBits ? top - kSelBits : 0;
                const unsigned dmask = (1u << (top - shift)) - 1u;
                const u64 fixed = prefix >> top;
                for (int i = tid; i < kSelBins; i += kSelThreads) hist[i] = 0u;
                __syncthreads();
                for (int i = tid; i < n; i += kSelThreads) {
                    const u64 key = buf[i];
                    if ((key >> top) == fixed) atomicAdd(&hist[(unsigned)(key >> shift) & dmask], 1u);
                }
                __syncthreads();
                pick(need);
                prefix |= (u64)s_digit << shift;
                need -= s_above;
                top = need == s_cnt ? 0 : shift;
            }
            best = reinterpret_cast<u64*>(hist);  // kSelBins words = 1024 keys >= k
            if (tid == 0) s_n = 0u;
            __syncthreads();
            for (int base = 0; base < n; base += kSelThreads) {
                const int i = base + tid;
                const u64 key = i < n ? buf[i] : 0ull;
                const bool p = i < n && key >= prefix;
                const unsigned b = __ballot_sync(kFullMask, p);
                unsigned at = 0;
                if (lane == 0 && b) at = atomicAdd(&s_n, (unsigned)__popc(b));
                at = __shfl_sync(kFullMask, at, 0);
                if (p) best[at + __popc(b & lanemask_lt())] = key;
            }
            __syncthreads();
            nb = k;
        }
        const int P = next_pow2(nb < 64 ? 64 : nb);  // <= 1024
        for (int j = nb + tid; j < P; j += kSelThreads) best[j] = 0ull;  // below every real key
        if (P <= 2 * kSelThreads)
            block_sort_reg_desc<u64, kSelThreads>(best, P);
        else
            block_sort_smem_desc(best, P);
        for (int j = tid; j < k; j += kSelThreads) {
            const u64 key = best[j];
            const unsigned col = 0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull);
            const unsigned u = (unsigned)(key >> 32);
            float v;
            if (u == 0x80000000u || u == 0xFFFFFFFFu)
                v = g.rp[col];  // -0.0 and NaN payloads: the input's bits
            else
                v = key_float(u);
            vals[(size_t)row * k + j] = v;
            idx[(size_t)row * k + j] = (int32_t)col;
        }
        __syncthreads();  // the buffer and histogram are reused by the next row
    }
}

}  // namespace

template <int L, bool kMask>
cudaError_t launch_stream(cudaStream_t s, const float* in, int rows, int cols, int k, float* vals, int32_t* idx,
                          unsigned* status, bool early, int flags, const uint8_t* keep, int32_t* row_count) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static int grid_cache[kMaxDev] = {};
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    if (device < 0 || device >= kMaxDev) return cudaErrorInvalidDevice;
    const void* fn = reinterpret_cast<const void*>(&topk_rows_stream_kernel<L, kMask>);
    int full;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (grid_cache[device] == 0) {
            int sms = 0, per_sm = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowRingBytes);
            if (e != cudaSuccess) return e;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kRowThreads, kRowRingBytes);
            if (e != cudaSuccess) return e;
            grid_cache[device] = sms * (per_sm < 1 ? 1 : per_sm);
        }
        full = grid_cache[device];
    }
    const int want = (rows + kRowWarps - 1) / kRowWarps;
    const int grid = want < full ? want : full;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kRowThreads);
    cfg.dynamicSmemBytes = kRowRingBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, topk_rows_stream_kernel<L, kMask>, in, rows, cols, k, vals, idx, status, flags,
                              keep, row_count);
}

// Rows of at most this many columns take the radix select (a row is read
// twice, the second time from L2); longer rows the streamed candidate
// buffer (one read).
constexpr int kSelMaxCols = 1 << 16;

cudaError_t rows_launch(cudaStream_t s, const float* in, int rows, int cols, int k, float* vals, int32_t* idx,
                        unsigned* status, bool early, int flags) {
    // k <= 128 streams rows (one warp per row); k > 128 takes one block per
    // row: a radix select for rows up to kSelMaxCols, else a streamed
    // shared-memory candidate buffer.
    const bool stream = k <= 128;
    const uint8_t* nk = nullptr;
    int32_t* nc = nullptr;
    if (stream && k <= 32) return launch_stream<1, false>(s, in, rows, cols, k, vals, idx, status, early, flags, nk, nc);
    if (stream && k <= 64) return launch_stream<2, false>(s, in, rows, cols, k, vals, idx, status, early, flags, nk, nc);
    if (stream) return launch_stream<4, false>(s, in, rows, cols, k, vals, idx, status, early, flags, nk, nc);
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static int grid_cache[kMaxDev][2] = {};
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    if (device < 0 || device >= kMaxDev) return cudaErrorInvalidDevice;
    int full, full_sel;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (grid_cache[device][0] == 0) {
            int sms = 0, per_sm = 0, per_sm_sel = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
            if (e != cudaSuccess) return e;
            const void* fn = reinterpret_cast<const void*>(&topk_rows_big_kernel);
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kBigRingBytes);
            if (e != cudaSuccess) return e;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kBigThreads, kBigRingBytes);
            if (e != cudaSuccess) return e;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &per_sm_sel, reinterpret_cast<const void*>(&topk_rows_select_kernel), kSelThreads, 0);
            if (e != cudaSuccess) return e;
            grid_cache[device][0] = sms * (per_sm < 1 ? 1 : per_sm);
            grid_cache[device][1] = sms * (per_sm_sel < 1 ? 1 : per_sm_sel);
        }
        full = grid_cache[device][0];
        full_sel = grid_cache[device][1];
    }
    if (cols <= kSelMaxCols) {
        const int grid = rows < full_sel ? rows : full_sel;
        topk_rows_select_kernel<<<grid, kSelThreads, 0, s>>>(in, rows, cols, k, vals, idx);
        return cudaGetLastError();
    }
    const int grid = rows < full ? rows : full;
    topk_rows_big_kernel<<<grid, kBigThreads, kBigRingBytes, s>>>(in, rows, cols, k, vals, idx, status);
    return cudaGetLastError();
}

bool rows_mask_aligned(const float* in, const uint8_t* keep) {
    // A row's 16-byte vectors start at element offsets congruent to -in/4
    // (mod 4); their keep words are 4-byte aligned when keep is congruent to
    // in/4 (mod 4).
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(keep);
    return (a & 3u) == 0 && ((b - (a >> 2)) & 3u) == 0;
}

cudaError_t rows_launch_masked(cudaStream_t s, const float* in, const uint8_t* keep, int rows, int cols, int k,
                               float* vals, int32_t* idx, int32_t* row_count, unsigned* status, bool early,
                               int flags) {
    if (k < 1 || k > 128 || !rows_mask_aligned(in, keep)) return cudaErrorInvalidValue;
    if (k <= 32) return launch_stream<1, true>(s, in, rows, cols, k, vals, idx, status, early, flags, keep, row_count);
    if (k <= 64) return launch_stream<2, true>(s, in, rows, cols, k, vals, idx, status, early, flags, keep, row_count);
    return launch_stream<4, true>(s, in, rows, cols, k, vals, idx, status, early, flags, keep, row_count);
}

}  // namespace topk
