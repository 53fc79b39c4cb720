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
// One block per row, 8 warps:
//   1. Every warp loads its first 4 KiB tile; each lane's maximum score key
//      is a group maximum.  The k-th largest of the 256 group maxima (at
//      least k elements reach it) becomes the row's start threshold.
//   2. Warps stream their tiles (128-bit loads, 8 in flight per lane) and
//      compare each float once against the threshold score; elements at or
//      above it get their exact 64-bit key, and keys above the warp's
//      threshold are compacted into a per-warp shared buffer.  A full
//      buffer is sorted and cut back to k, raising the warp's threshold,
//      which is shared with the other warps through shared memory.
//   3. The warps' sorted lists are merged pairwise (bitonic), and the k best
//      keys give the columns; values are re-read from the row so their bits
//      are the input's.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "topk_device.cuh"
#include "topk_internal.h"

namespace topk {

namespace {

constexpr int kU = 8;              // 16-byte loads in flight per lane
constexpr int kTileVec = 32 * kU;  // float4 vectors per warp-tile
constexpr int kWarps = 8;

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

// Elements that may beat threshold score tf: v >= tf, or v is NaN.
__device__ __forceinline__ bool maybe(float v, float tf) { return !(v < tf); }

__device__ __forceinline__ float4 ld4(const float4* p) { return __ldg(p); }

struct RowBufT {
    u64* buf;
    int cnt;
    u64 T;  // only keys > T are admitted
};

template <int B>
__device__ __forceinline__ void rows_admit(RowBufT& w, float v, unsigned col, float tf, int lane) {
    bool p = false;
    u64 key = 0;
    if (maybe(v, tf)) {
        key = full_key(v, col);
        p = key > w.T;
    }
    const unsigned m = __ballot_sync(kFullMask, p);
    if (p) w.buf[w.cnt + __popc(m & lanemask_lt())] = key;
    w.cnt += __popc(m);
}

// Sort the buffer, keep the k best keys, raise T to the k-th.  Returns true
// when T was raised.
template <int B>
__device__ bool rows_flush(RowBufT& w, int k, int lane) {
    __syncwarp();
    bool raised = false;
    for (int p = w.cnt + lane; p < B; p += 32) w.buf[p] = 0ull;
    __syncwarp();
    warp_sort_smem_desc(w.buf, B, lane);
    if (w.cnt >= k) {
        const u64 kth = w.buf[k - 1];
        if (kth > w.T) {
            w.T = kth;
            raised = true;
        }
    }
    w.cnt = w.cnt < k ? w.cnt : k;
    __syncwarp();
    return raised;
}

template <int B>
__global__ void __launch_bounds__(kWarps * 32, 1)
topk_rows_smem_kernel(const float* __restrict__ in, int cols, int k, float* __restrict__ vals,
                      int32_t* __restrict__ idx) {
    extern __shared__ __align__(16) u64 smem64[];
    __shared__ u64 s_T;
    __shared__ unsigned s_gmax[kWarps * 32];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const size_t row = blockIdx.x;
    const float* rp = in + row * (size_t)cols;

    // Row split: unaligned head (< 4), 16-byte aligned float4 body, tail.
    const uintptr_t addr = reinterpret_cast<uintptr_t>(rp);
    int head = (int)(((16u - (unsigned)(addr & 15u)) & 15u) >> 2);
    if (head > cols) head = cols;
    const float4* body = reinterpret_cast<const float4*>(rp + head);
    const int nvec = (cols - head) >> 2;
    const int tail0 = head + nvec * 4;
    const int ntiles = (nvec + kTileVec - 1) / kTileVec;

    RowBufT w{smem64 + warp * B, 0, 0ull};

    // 1. First tile of each warp: group maxima -> start threshold.
    float4 r[kU];
    const int t0 = warp;
    auto load = [&](int tile) {
        const int base = tile * kTileVec + lane;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = base + u * 32;
            r[u] = (tile < ntiles && i < nvec) ? ld4(body + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    load(t0);
    {
        unsigned gm = 0u;  // key 0 is below every real key
        if (t0 < ntiles) {
            const int base = t0 * kTileVec + lane;
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (base + u * 32 < nvec) {
                    gm = max(gm, score_key(__float_as_uint(r[u].x)));
                    gm = max(gm, score_key(__float_as_uint(r[u].y)));
                    gm = max(gm, score_key(__float_as_uint(r[u].z)));
                    gm = max(gm, score_key(__float_as_uint(r[u].w)));
                }
            }
        }
        s_gmax[threadIdx.x] = gm;
    }
    if (threadIdx.x == 0) s_T = 0ull;
    __syncthreads();
    if (warp == 0 && k <= kWarps * 32) {
        unsigned g[kWarps];
#pragma unroll
        for (int j = 0; j < kWarps; ++j) g[j] = s_gmax[j * 32 + lane];
        warp_sort_desc<kWarps>(g, lane);
        const unsigned seed = warp_sorted_at<kWarps>(g, k - 1);
        if (lane == 0) s_T = (u64)seed << 32;  // admits every key with score >= seed
    }
    __syncthreads();
    w.T = s_T;

    // Scalars outside the aligned body: taken by warp 0.
    if (warp == 0) {
        const int ns = head + (cols - tail0);
        const int col = lane < head ? lane : tail0 + (lane - head);
        const float v = lane < ns ? rp[col] : 0.f;
        const float tf = key_float((unsigned)(w.T >> 32));
        bool p = false;
        u64 key = 0;
        if (lane < ns && maybe(v, tf)) {
            key = full_key(v, (unsigned)col);
            p = key > w.T;
        }
        const unsigned m = __ballot_sync(kFullMask, p);
        if (p) w.buf[w.cnt + __popc(m & lanemask_lt())] = key;
        w.cnt += __popc(m);
    }

    // 2. Stream the row.
    for (int tile = t0; tile < ntiles; tile += kWarps) {
        if (tile != t0) load(tile);
        w.T = kmax(w.T, *(volatile u64*)&s_T);
        const float tf = key_float((unsigned)(w.T >> 32));
        bool any = false;
#pragma unroll
        for (int u = 0; u < kU; ++u)
            any |= maybe(r[u].x, tf) | maybe(r[u].y, tf) | maybe(r[u].z, tf) | maybe(r[u].w, tf);
        if (__any_sync(kFullMask, any)) {
            const int base = tile * kTileVec + lane;
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (w.cnt > B - 128) {
                    if (rows_flush<B>(w, k, lane) && lane == 0) atomicMax(&s_T, w.T);
                }
                const float tfu = key_float((unsigned)(w.T >> 32));
                const int vi = base + u * 32;
                const bool valid = vi < nvec;
                const unsigned c0 = (unsigned)(head + vi * 4);
                rows_admit<B>(w, r[u].x, c0 + 0, valid ? tfu : __int_as_float(0x7f800000), lane);
                rows_admit<B>(w, r[u].y, c0 + 1, valid ? tfu : __int_as_float(0x7f800000), lane);
                rows_admit<B>(w, r[u].z, c0 + 2, valid ? tfu : __int_as_float(0x7f800000), lane);
                rows_admit<B>(w, r[u].w, c0 + 3, valid ? tfu : __int_as_float(0x7f800000), lane);
            }
        }
    }

    // 3. Per-warp sorted lists, block merge, output.
    if (rows_flush<B>(w, k, lane) && lane == 0) atomicMax(&s_T, w.T);
    const int K = next_pow2(k < 32 ? 32 : k);
    for (int p = w.cnt + lane; p < K; p += 32) w.buf[p] = 0ull;
#pragma unroll 1
    for (int s = 1; s < kWarps; s <<= 1) {
        __syncthreads();
        if ((warp & (2 * s - 1)) == 0) {
            u64* a = smem64 + warp * B;
            const u64* b = smem64 + (warp + s) * B;
            for (int i = lane; i < K; i += 32) a[i] = kmax(a[i], b[K - 1 - i]);
            __syncwarp();
            warp_merge_smem_desc(a, K, lane);
        }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
        const u64 key = smem64[j];
        const unsigned col = 0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull);
        // Every key in the merged list is a real element (at least k elements
        // reach the start threshold), so col < cols; the guard only keeps a
        // broken invariant from turning into an out-of-row read.
        vals[row * (size_t)k + j] = col < (unsigned)cols ? __ldg(rp + col) : __int_as_float(0x7fc00000);
        idx[row * (size_t)k + j] = (int32_t)col;
    }
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

cudaError_t rows_launch(cudaStream_t s, const float* in, int rows, int cols, int k, float* vals, int32_t* idx,
                        unsigned* status, bool early, int flags) {
    // k <= 128 streams rows (one warp per row); k > 128 uses one block per row
    // with shared-memory buffers.
    const bool stream = k <= 128;
    const uint8_t* nk = nullptr;
    int32_t* nc = nullptr;
    if (stream && k <= 32) return launch_stream<1, false>(s, in, rows, cols, k, vals, idx, status, early, flags, nk, nc);
    if (stream && k <= 64) return launch_stream<2, false>(s, in, rows, cols, k, vals, idx, status, early, flags, nk, nc);
    if (stream) return launch_stream<4, false>(s, in, rows, cols, k, vals, idx, status, early, flags, nk, nc);
    const size_t smem = (size_t)kWarps * 2048 * sizeof(u64);
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&topk_rows_smem_kernel<2048>),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (k <= 128) {
        const size_t smem256 = (size_t)kWarps * 256 * sizeof(u64);
        topk_rows_smem_kernel<256><<<rows, kWarps * 32, smem256, s>>>(in, cols, k, vals, idx);
    } else {
        topk_rows_smem_kernel<2048><<<rows, kWarps * 32, smem, s>>>(in, cols, k, vals, idx);
    }
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
