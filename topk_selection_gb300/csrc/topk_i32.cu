// int32 TopK: the k largest values of a large array, sorted descending.
//
// Method ("CUDA parallel optimisation: TopK, shared memory and two-stage
// reduction"): section 2.1 -- every block reduces its share of the input to
// k candidates (grid-stride loop, per-thread local top-k, shared-memory tree
// merge); section 2.2 -- a second single-block pass over the grid*k
// candidates gives the final k, identical to the CPU's answer.
//
// What is kept and what differs on sm_103a:
//   * Stage 1 streams 4 KiB tiles with bulk copies (cp.async.bulk, three in
//     flight per warp into the warp's own shared-memory ring) in a
//     persistent grid of one block per SM (15 consumer warps, one monitor
//     warp, 112 registers a thread: measured faster than two blocks of 8
//     consumers at 96 registers, which spilled).  Instead of an insertion sort per
//     element, each warp compares every element once against a running
//     threshold t; the rare survivors are compacted (ballot + popc) into a
//     per-warp shared-memory queue and merged 32 at a time into the warp's
//     sorted top-K list, which it keeps in registers (bitonic sort of the 32,
//     then a bitonic merge; the warp-shuffle technique of "Complete guide to
//     CUDA reduction optimisation").
//   * Thresholds.  Any t used to discard is a value with at least k input
//     elements >= t, and every such t is published (atomicMax) to one global
//     word before the block finishes.  Sources of t:
//       - the warp's own k-th largest once its list holds k values;
//       - a start value: the k-th largest of 32*G group maxima of the warp's
//         first tile, and of the array's last 256 (k > 64: 512) elements (so that sorted
//         ascending input stays cheap);
//       - each block keeps its running maximum in a global slot; the k-th
//         largest of all blocks' maxima is a valid t (k distinct blocks each
//         hold an element that large), and once every block has streamed a
//         little it sits close to the true k-th value of the whole input.
//         One warp per block refreshes it each round, in turn.
//   * The block merge (section 2.1's tree) is warp 0 merging the other
//     warps' sorted lists into its own, bitonically.
//   * The second pass (section 2.2) runs in the same launch: the last block
//     to finish (atomic ticket, no waiting) selects the answer from the
//     grid*k candidates.  With t_g the final global threshold, the answer is
//     the candidates greater than t_g, sorted, padded with copies of t_g
//     when fewer than k exceed it.  If more candidates exceed t_g than fit in
//     shared memory, an 8-bit-digit radix select (the per-digit histogram of
//     "GPU radix sort", histogram section) finds the exact k-th value first.
//   * The last block zeroes the control words and the block-maximum slots,
//     so the next launch on the same scratch starts clean.  No block ever
//     waits on another.
//   * k > 128 uses the radix select of topk_radix.cu instead.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "topk_device.cuh"
#include "topk_internal.h"

namespace topk {

namespace {

constexpr int kU = 8;              // 16-byte loads in flight per lane
constexpr int kTileVec = 32 * kU;  // int4 vectors per warp-tile (4 KiB)
constexpr int kQueue = 256;        // per-warp survivor queue (>= 31 + 128)

__device__ __forceinline__ unsigned bias(int v) { return (unsigned)v ^ 0x80000000u; }
__device__ __forceinline__ int unbias(unsigned u) { return (int)(u ^ 0x80000000u); }

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int max4(int4 v) { return kmax(kmax(v.x, v.y), kmax(v.z, v.w)); }

struct Scratch {
    unsigned* status;  // sticky error bits (kStatusWaitTimeout)
    I32Ctrl* ctrl;
    unsigned* bmax;    // per-block running maxima, biased
    unsigned char* dyn;  // tile-claim counters, one per kI32DynStride bytes
    int32_t* counts;   // per list: entries above the grid threshold at the block's end
    int32_t* tmax;     // per tile: its maximum (grids with fewer blocks than k)
    int32_t* cand;     // per block: its sorted candidate lists
};

__device__ __forceinline__ Scratch scratch_view(unsigned char* base) {
    return Scratch{reinterpret_cast<unsigned*>(base + kI32StatusOffset), reinterpret_cast<I32Ctrl*>(base + kI32CtrlOffset),
                   reinterpret_cast<unsigned*>(base + kI32BmaxOffset), base + kI32DynOffset,
                   reinterpret_cast<int32_t*>(base + kI32CountOffset),
                   reinterpret_cast<int32_t*>(base + kI32TileMaxOffset),
                   reinterpret_cast<int32_t*>(base + kI32CandOffset)};
}

__device__ __forceinline__ unsigned* dyn_counter(const Scratch& sc, int c) {
    return reinterpret_cast<unsigned*>(sc.dyn + (size_t)c * kI32DynStride);
}

// Input split: an unaligned head (< 4 elements), a 16-byte aligned body of
// int4 vectors, a scalar tail (< 4 elements).
struct Split {
    size_t head, nvec, tail0, ntiles;
    const int4* body;
};

__device__ __forceinline__ Split split_input(const int32_t* in, size_t n) {
    Split s;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(in);
    s.head = ((16u - (unsigned)(addr & 15u)) & 15u) >> 2;
    if (s.head > n) s.head = n;
    s.body = reinterpret_cast<const int4*>(in + s.head);
    s.nvec = (n - s.head) >> 2;
    s.tail0 = s.head + s.nvec * 4;
    s.ntiles = (s.nvec + kTileVec - 1) / kTileVec;
    return s;
}

// k-th largest of the warp's 32*GL group maxima (each group a disjoint set of
// real elements, so at least k input elements are >= the result).  Groups
// made only of padding have maximum INT_MIN, which is always a valid bound.
template <int GL, int NV>
__device__ __forceinline__ int seed_from_groups(const int4 (&r)[NV], int k, int lane) {
    static_assert(NV % GL == 0, "groups must split the lane's vectors evenly");
    int g[GL];
#pragma unroll
    for (int j = 0; j < GL; ++j) {
        int m = INT_MIN;
#pragma unroll
        for (int u = j * (NV / GL); u < (j + 1) * (NV / GL); ++u) m = kmax(m, max4(r[u]));
        g[j] = m;
    }
    warp_sort_desc<GL>(g, lane);
    return warp_sorted_at<GL>(g, k - 1);
}

// Append the lanes' values that exceed t to q[*nq...] (warp-uniform count).
__device__ __forceinline__ void enqueue(int* q, int& nq, int v, int t, int lane) {
    const bool p = v > t;
    const unsigned m = __ballot_sync(kFullMask, p);
    if (p) q[nq + __popc(m & lanemask_lt())] = v;
    nq += __popc(m);
}


// The k-th largest (1 <= k) of the unsigned values that the block's threads
// hold, N per thread (pad with 0): an 8-bit-digit radix select ("GPU radix
// sort", histogram section), most significant digit first, four rounds of
// a shared 256-bin histogram.  Every thread must call it; every thread
// gets the result.  With fewer than k values in all, the result is 0.
template <int N>
__device__ unsigned block_kth_largest(const unsigned (&v)[N], unsigned k, unsigned* hist, unsigned* pick) {
    const int lane = threadIdx.x & 31;
    unsigned prefix = 0, need = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        const unsigned mask = shift == 24 ? 0u : 0xFFFFFFFFu << (shift + 8);
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
        if (threadIdx.x == 0) pick[0] = 0u, pick[1] = need;
        __syncthreads();
#pragma unroll
        for (int q = 0; q < N; ++q)
            if ((v[q] & mask) == prefix) atomicAdd(&hist[(v[q] >> shift) & 255u], 1u);
        __syncthreads();
        if (threadIdx.x < 32) {
            unsigned cnt[8], tot = 0;
#pragma unroll
            for (int b = 0; b < 8; ++b) tot += (cnt[b] = hist[lane * 8 + b]);
            unsigned x = tot;  // sum over this lane and the lanes above (higher bins)
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_down_sync(kFullMask, x, o);
                if (lane + o < 32) x += y;
            }
            unsigned acc = x - tot;  // values in higher bins
            if (acc < need && need <= acc + tot) {
#pragma unroll
                for (int b = 7; b >= 0; --b) {
                    if (acc + cnt[b] >= need) {
                        pick[0] = (unsigned)(lane * 8 + b);
                        pick[1] = need - acc;
                        break;
                    }
                    acc += cnt[b];
                }
            }
        }
        __syncthreads();
        prefix |= pick[0] << shift;
        need = pick[1];
        __syncthreads();
    }
    return prefix;
}

constexpr int kLongLists = 64;  // second stage: lists whose survivors the block reads together

// One warp: sort list[0, nlist) (nlist <= 32*N) descending in registers and
// write out[0, k): the sorted entries, then copies of T; in the kind's words.
template <int N, int KIND>
__device__ __forceinline__ void warp_sort_out(const int* list, int nlist, int k, int T, int32_t* out, int lane) {
    int v[N];
#pragma unroll
    for (int j = 0; j < N; ++j) {
        const int p = j * 32 + lane;
        v[j] = p < nlist ? list[p] : INT_MIN;
    }
    warp_sort_desc<N>(v, lane);
#pragma unroll
    for (int j = 0; j < N; ++j) {
        const int p = j * 32 + lane;
        if (p < k) out[p] = ordered<KIND>(p < nlist ? v[j] : T);
    }
    for (int p = 32 * N + lane; p < k; p += 32) out[p] = ordered<KIND>(T);
}

// ---------------------------------------------------------------- stage 2 --
//
// Every block leaves `lists_per_block` sorted lists of K entries (INT_MIN
// padded) in its candidate area, and for each list the number of leading
// entries that exceed the grid threshold it read when it finished.  The
// entries after that count are at most a published threshold, so they can
// never be needed: only the counted prefixes are gathered.

// Run by the last block to finish.  `room` ints of shared memory at `list`;
// cap_limit > 0 lowers the list capacity (to exercise the radix-select path).
template <int KIND>
__device__ void second_stage(const Scratch& sc, int k, int lists_per_block, int K, int32_t* __restrict__ out,
                             int* list, int room, int cap_limit, int* s_count, int ntmax) {
    const int lane = threadIdx.x & 31;
    __shared__ unsigned s_hist[256];
    __shared__ unsigned s_pick[2];
    // Every other block's writes are visible here: thread 0 drew the last
    // ticket with acquire semantics, and the barrier after it orders this
    // block's reads after that.
    int tg = unbias(ld_relaxed_gpu(&sc.ctrl->thresh));
    const int nlists = (int)gridDim.x * lists_per_block;
    // Each list's count and its first four entries, loaded together (one
    // round trip for the usual case of at most four survivors per list).
    // Lists and tile maxima: at most kBatch per thread.
    constexpr int kBatch = kI32MaxTileMax / 256;
    int c[kBatch];
    int4 h[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
        const int l = q * (int)blockDim.x + (int)threadIdx.x;
        c[q] = l < nlists ? __ldcg(sc.counts + l) : 0;
        h[q] = l < nlists ? __ldcg(reinterpret_cast<const int4*>(sc.cand + (size_t)l * K))
                          : make_int4(INT_MIN, INT_MIN, INT_MIN, INT_MIN);
    }
    // The list is bitonic-sorted in place at a power-of-two length, so its
    // capacity is the largest power of two that fits.
    int cap = 1;
    while (2 * cap <= room) cap *= 2;
    if (cap_limit > 0 && cap_limit < cap) cap = cap_limit;
    if (cap < k) cap = k;  // the sorted list must be able to hold the answer

    // Before gathering: when the lists' counts (entries above each block's
    // threshold at its end, so at least as many as will pass) add up to more
    // than one warp's sort (256), tighten tg with a bound of the gather's
    // own, so that each list yields few entries: with at least k lists, the
    // k-th largest list head (each list starts with its block's maximum, and
    // k distinct blocks hold an element that large); with fewer blocks than
    // k, the k-th largest tile maximum (k distinct tiles).  Both are valid
    // thresholds however little the blocks learnt from each other while
    // streaming (a launch that started early, a short input).
    {
        int cs = 0;
#pragma unroll
        for (int q = 0; q < kBatch; ++q) cs += c[q];
        cs = __reduce_add_sync(kFullMask, cs);
        if (threadIdx.x == 0) *s_count = 0;
        __syncthreads();
        if (lane == 0 && cs) atomicAdd(s_count, cs);
        __syncthreads();
    }
    if (*s_count > 256 && (nlists >= k || ntmax >= k)) {
        unsigned v[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int l = q * (int)blockDim.x + (int)threadIdx.x;
            if (ntmax >= k)  // tiles, when recorded, outnumber blocks eightfold
                v[q] = l < ntmax ? bias(__ldcg(sc.tmax + l)) : 0u;
            else
                v[q] = bias(h[q].x);
        }
        tg = kmax(tg, unbias(block_kth_largest<kBatch>(v, (unsigned)k, s_hist, s_pick)));
    }
    __syncthreads();
    // Each thread takes its lists' first four entries; a list whose fourth
    // entry still exceeds tg is queued, and the block reads the rest of the
    // queued lists together (a single list can hold up to K survivors, e.g.
    // the last block of an ascending input).
    __shared__ int2 s_long[kLongLists];
    __shared__ int s_nlong;
    if (threadIdx.x == 0) *s_count = 0, s_nlong = 0;
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
        const int l = q * (int)blockDim.x + (int)threadIdx.x;
        const int head[4] = {h[q].x, h[q].y, h[q].z, h[q].w};
        int p = 0;
#pragma unroll
        for (; p < 4; ++p) {
            if (p >= c[q] || head[p] <= tg) break;  // the list is sorted: nothing after this exceeds tg
            const int pos = atomicAdd(s_count, 1);
            if (pos < cap) list[pos] = head[p];
        }
        if (p == 4 && c[q] > 4) {
            const int slot = atomicAdd(&s_nlong, 1);
            if (slot < kLongLists) {
                s_long[slot] = make_int2(l, c[q]);
            } else {  // too many long lists to queue: this thread reads the rest
                const int32_t* src = sc.cand + (size_t)l * K;
                for (int pp = 4; pp < c[q]; ++pp) {
                    const int v = __ldcg(src + pp);
                    if (v <= tg) break;
                    const int pos = atomicAdd(s_count, 1);
                    if (pos < cap) list[pos] = v;
                }
            }
        }
    }
    __syncthreads();
    // The queued lists' entries after the fourth, as one flat range read by
    // the whole block: s_lstart[j] is where list j starts in that range.
    // Skipped, code and all, when no list was queued (the usual case).
    __shared__ int s_lstart[kLongLists + 1];
    const int nlong = s_nlong < kLongLists ? s_nlong : kLongLists;
    if (nlong > 0) {
    if (threadIdx.x < 32) {
        int run = 0;
        for (int j0 = 0; j0 < nlong; j0 += 32) {
            const int j = j0 + lane;
            const int len = j < nlong ? s_long[j].y - 4 : 0;
            int x = len;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFullMask, x, o);
                if (lane >= o) x += y;
            }
            if (j < nlong) s_lstart[j] = run + x - len;
            run += __shfl_sync(kFullMask, x, 31);
        }
        if (lane == 0) s_lstart[nlong] = run;
    }
    __syncthreads();
    const int flat = s_lstart[nlong];
    constexpr int kFlatU = 4;  // loads in flight per thread
    for (int e0 = (int)threadIdx.x; e0 < flat; e0 += kFlatU * (int)blockDim.x) {
        int v[kFlatU];
#pragma unroll
        for (int u = 0; u < kFlatU; ++u) {
            const int e = e0 + u * (int)blockDim.x;
            v[u] = INT_MIN;
            if (e < flat) {
                int lo = 0, hi = nlong - 1;  // the list holding e: last j with s_lstart[j] <= e
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_lstart[mid] <= e) lo = mid; else hi = mid - 1;
                }
                v[u] = __ldcg(sc.cand + (size_t)s_long[lo].x * K + 4 + (e - s_lstart[lo]));
            }
        }
#pragma unroll
        for (int u = 0; u < kFlatU; ++u) {
            const int e = e0 + u * (int)blockDim.x;
            if (e < flat && v[u] > tg) {
                const int pos = atomicAdd(s_count, 1);
                if (pos < cap) list[pos] = v[u];
            }
        }
    }
    __syncthreads();
    }
    const int above = *s_count;

    int T = tg;         // value that fills the places after the sorted list
    int nlist = above;  // sorted entries that come first
    if (above > cap) {
        // Radix select over every candidate above tg: the exact k-th largest
        // value T, most significant 8-bit digit first.
        __shared__ unsigned hist[256];
        __shared__ unsigned s_prefix, s_need;
        const size_t M = (size_t)nlists * K;
        const size_t Mr = (M + blockDim.x - 1) / blockDim.x * blockDim.x;
        unsigned prefix = 0, pmask = 0, need = (unsigned)k;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
            __syncthreads();
            for (size_t i = threadIdx.x; i < M; i += blockDim.x) {
                const int v = __ldcg(sc.cand + i);
                const unsigned u = bias(v);
                if (v > tg && (u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                unsigned acc = 0;
                int d = 255;
                for (; d > 0; --d) {
                    if (acc + hist[d] >= need) break;
                    acc += hist[d];
                }
                s_prefix = prefix | ((unsigned)d << shift);
                s_need = need - acc;
            }
            __syncthreads();
            prefix = s_prefix;
            need = s_need;
            pmask |= 255u << shift;
            __syncthreads();
        }
        T = unbias(prefix);
        // Values strictly above T: fewer than k of them.
        if (threadIdx.x == 0) *s_count = 0;
        __syncthreads();
        for (size_t i = threadIdx.x; i < Mr; i += blockDim.x) {
            const int v = i < M ? __ldcg(sc.cand + i) : INT_MIN;
            const bool p = v > T;
            const unsigned m = __ballot_sync(kFullMask, p);
            int base = 0;
            if (lane == 0 && m) base = atomicAdd(s_count, __popc(m));
            base = __shfl_sync(kFullMask, base, 0);
            if (p) list[base + __popc(m & lanemask_lt())] = v;
        }
        __syncthreads();
        nlist = *s_count;
    }

    if (nlist <= 32) {
        // At most 32: one warp sorts them in registers.
        if (threadIdx.x < 32) warp_sort_out<1, KIND>(list, nlist, k, T, out, lane);
    } else if (nlist <= 512) {
        // Up to 512: every entry's place is the number of entries above it
        // (equal entries ordered by their slot), one pass over the list in
        // shared memory and no barrier.  This code runs once, after the
        // input stream has pushed it out of L2: a small loop beats an
        // unrolled sorting network here (measured at 1e8, k = 100, 146
        // entries: warp network 6.9 us, block network 4.1 us).
        for (int i = threadIdx.x; i < nlist; i += blockDim.x) {
            const int v = list[i];
            int r = 0;
            for (int j = 0; j < nlist; ++j) {
                const int x = list[j];
                r += (x > v || (x == v && j < i)) ? 1 : 0;
            }
            if (r < k) out[r] = ordered<KIND>(v);
        }
        for (int i = nlist + threadIdx.x; i < k; i += blockDim.x) out[i] = ordered<KIND>(T);
    } else {
        // The block sorts them in shared memory (rolled loops).
        const int L = next_pow2(nlist);
        for (int i = nlist + threadIdx.x; i < L; i += blockDim.x) list[i] = INT_MIN;
        block_sort_smem_desc(list, L);
        for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = ordered<KIND>(i < nlist ? list[i] : T);
    }
    // Leave the scratch as the next launch expects it.
    for (int i = threadIdx.x; i < (int)gridDim.x; i += blockDim.x) sc.bmax[i] = 0u;
    for (int c = threadIdx.x; c < kI32DynRanges; c += blockDim.x) *dyn_counter(sc, c) = 0u;
    if (threadIdx.x == 0) {
        sc.ctrl->thresh = 0u;
        sc.ctrl->ticket = 0u;
    }
}

// Publish this block's threshold and take a ticket (after every thread has
// written its candidates); returns true in the last block to finish.
// The ticket is an acquire-release atomic: its release makes the block's
// candidate writes (ordered before it by the barrier) and the threshold
// published just before it visible to the block that draws the last
// ticket, whose acquire orders its later reads after them.
__device__ __forceinline__ unsigned ticket_acq_rel(unsigned* p) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
    return old;
}

__device__ __forceinline__ bool block_done(const Scratch& sc, int block_thresh, int* s_last) {
    __syncthreads();
    if (threadIdx.x == 0) {
        if (block_thresh != INT_MIN) atomicMax(&sc.ctrl->thresh, bias(block_thresh));
        const unsigned ticket = ticket_acq_rel(&sc.ctrl->ticket);
        *s_last = ticket == gridDim.x - 1;
    }
    __syncthreads();
    return *s_last != 0;
}

// Write a warp's sorted K-list (lst[j] at position j*32 + lane) and the
// number of its leading entries above t_now.
template <int L>
__device__ __forceinline__ void write_list(const Scratch& sc, int list_id, const int (&lst)[L], int t_now, int lane) {
    int32_t* dst = sc.cand + (size_t)list_id * (32 * L);
    int count = 0;
#pragma unroll
    for (int j = 0; j < L; ++j) {
        dst[j * 32 + lane] = lst[j];
        count += __popc(__ballot_sync(kFullMask, lst[j] > t_now));
    }
    if (lane == 0) sc.counts[list_id] = count;
}

// ------------------------------------------------- k <= 128: register lists --

template <int L>
using WarpList = RegList<L, int>;

// Streaming: every consumer warp owns a ring of kWarpStages shared-memory
// stages of one 4 KiB tile each and keeps bulk copies of its own next tiles
// in flight; as soon as a tile is in registers the warp re-arms that stage
// with the copy of its tile kWarpStages steps ahead.  No warp ever waits for
// another warp's progress.  Consumers touch only shared memory; a monitor
// warp carries thresholds between the block and the grid.
constexpr int kCons = 15;                    // consumer warps per block (one block per SM)
constexpr int kMonitor = kCons;              // warp index of the monitor
constexpr int kStreamThreads = (kCons + 1) * 32;
constexpr int kWarpStages = 3;               // tiles in flight per consumer warp
constexpr int kRingBytes = kCons * kWarpStages * kTileVec * 16;
constexpr int kMonitorRounds = 1 << 20;      // bound on the monitor's polling rounds
constexpr int kStaticPct = 100;              // share of the input assigned up front (percent)
static_assert(kStreamThreads * (kI32MaxTileMax / 256) >= kI32MaxTileMax &&
                  kStreamThreads * (kI32MaxTileMax / 256) >= kI32MaxGrid,
              "second stage: every list and tile maximum has a thread slot");

template <int L, int GL, int KIND>
// 112 registers a thread (no spills); with 16 warps a block, one block per SM.
__global__ void __maxnreg__(112)
topk_i32_stream_kernel(const int32_t* __restrict__ in, size_t n, int k, int32_t* __restrict__ out,
                       unsigned char* __restrict__ scratch, int cap_limit, int release, int static_pct) {
    constexpr int K = 32 * L;
    extern __shared__ __align__(128) int4 ring[];             // per-warp stages; later the stage-2 list
    __shared__ __align__(16) int s_queue[kCons * kQueue];      // survivor queues, then the merge area
    __shared__ int s_sel[256];                                 // monitor: block maxima above t
    __shared__ __align__(8) uint64_t full_bar[kCons * kWarpStages];
    __shared__ int s_thresh, s_cmax, s_done, s_last, s_count;
    __shared__ int s_tile[kCons * kWarpStages];                // tile id of each stage's copy

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const Scratch sc = scratch_view(scratch);
    if (threadIdx.x == 0) {
        s_thresh = INT_MIN;
        s_cmax = INT_MIN;
        s_done = 0;
        for (int s = 0; s < kCons * kWarpStages; ++s) mbar_init(&full_bar[s], 1);
        mbar_init_fence();
    }
    __syncthreads();

    const Split sp = split_input(in, n);
    const size_t G = gridDim.x;
    const size_t b = blockIdx.x;
    // Work schedule, in items of at most one 4 KiB tile (kTileVec vectors).
    // With P = G*kCons consumer warps, warp p = b + G*w (interleaved, so
    // that neighbouring warps read neighbouring tiles at the same time):
    //   full rounds   round i < R: item p + P*i, the tile of that index;
    //   piece         item R*P + p: the warp's equal share (to one vector)
    //                 of the vectors left of the static part after the full
    //                 rounds, so that every warp streams the same bytes;
    //   claimed       the vectors after the static part (a share of
    //                 100 - static_pct percent) as tiles in nr contiguous
    //                 ranges with a claim counter each; a warp that has
    //                 finished its static items claims one tile at a time,
    //                 from its own range first, then from any range with
    //                 tiles left.
    // Item ids fit 31 bits: n <= 2^40 elements is at most 2^30 tiles.  By
    // default (static_pct = 100), and always with fewer blocks than k, items
    // are whole tiles only: rounds up to the last tile, no pieces, nothing
    // claimed.  (Measured on GB300 at 1e8: equal pieces and claimed tiles
    // both finished later than whole tiles; the warps' rates differ more
    // than their shares.)  With fewer blocks than k the k-th largest tile
    // maximum bounds the answer in the second stage.
    const unsigned ntiles = (unsigned)sp.ntiles;
    // Tile maxima, when the grid has fewer than 2k blocks (their k-th
    // largest maximum is then a weak bound) and the input is small enough.
    // Writing them waits for the previous launch first (it may still read
    // its own), so they stay off where early start pays.
    const bool use_tmax = (int)G < 2 * k && ntiles <= (unsigned)kI32MaxTileMax;
    // All static (the default): whole tiles round-robin, as many rounds as
    // it takes, no pieces and nothing claimed.
    const bool whole = use_tmax || static_pct >= 100;
    const unsigned P = (unsigned)G * kCons;
    const size_t S_vec = whole ? sp.nvec : sp.nvec * (size_t)static_pct / 100;  // static vectors
    const unsigned R = whole ? (ntiles + P - 1) / P : (unsigned)(S_vec / ((size_t)P * kTileVec));
    const size_t full_vec = whole ? sp.nvec : (size_t)R * P * kTileVec;  // vectors of the full rounds
    const size_t rem = S_vec > full_vec ? S_vec - full_vec : 0;             // vectors of the pieces (< P tiles)
    const unsigned piece_q = (unsigned)(rem / P), piece_r = (unsigned)(rem % P);
    const bool pieces = rem > 0;
    const unsigned D = (unsigned)((sp.nvec - S_vec + kTileVec - 1) / kTileVec);  // claimed tiles
    const int nr = D < (unsigned)kI32DynRanges ? (int)D : kI32DynRanges;
    const unsigned dyn_id0 = R * P + (pieces ? P : 0u);  // id of the first claimed tile
    // Vectors [base, base + cnt) of item `id` (cnt 0: nothing there).
    auto item_span = [&](unsigned id, size_t& base, unsigned& cnt) {
        if (id < R * P) {
            base = (size_t)id * kTileVec;
        } else if (id < dyn_id0) {
            const unsigned q = id - R * P;
            base = full_vec + (size_t)q * piece_q + (q < piece_r ? q : piece_r);
            cnt = piece_q + (q < piece_r ? 1u : 0u);
            return;
        } else {
            base = S_vec + (size_t)(id - dyn_id0) * kTileVec;
        }
        cnt = base >= sp.nvec ? 0u : (sp.nvec - base < (size_t)kTileVec ? (unsigned)(sp.nvec - base) : (unsigned)kTileVec);
    };
    // The block-maxima threshold needs at least k blocks.
    const bool use_bmax = (int)G >= k;

    WarpList<L> wl;
    wl.init(INT_MIN);

    if (warp == kMonitor) {
        // Start value from the array's last 256 (k > 64: 512) elements (keeps sorted
        // ascending input cheap), then poll: publish the block's threshold
        // and maximum, pull the grid's threshold and the k-th largest block
        // maximum.  Every value it puts in s_thresh is a valid threshold.
        {
            // The tail sample: TV vectors per lane, so that its 32*GL groups
            // of whole vectors are at least k.
            constexpr int TV = GL > 2 ? GL : 2;
            if (sp.nvec > 0) {
                int4 s[TV];
                const long long tv = (long long)sp.nvec - 32 * TV + TV * lane;
#pragma unroll
                for (int q = 0; q < TV; ++q)
                    s[q] = tv + q >= 0 ? ordered4<KIND>(__ldg(sp.body + tv + q)) : make_int4(INT_MIN, INT_MIN, INT_MIN, INT_MIN);
                const int tseed = seed_from_groups<GL>(s, k, lane);
                if (lane == 0) atomicMax(&s_thresh, tseed);
            }
        }
        // The scratch is the previous launch's until it completes (this
        // kernel may start early, see the host side): wait for it here.
        grid_dependency_wait();
        int pub_t = INT_MIN, pub_cmax = INT_MIN;
        for (int round = 0; round < kMonitorRounds; ++round) {
            // Once every consumer is done the block publishes its own
            // threshold with its ticket: nothing is left for the monitor.
            if (*(volatile int*)&s_done == kCons) break;
            const int st = *(volatile int*)&s_thresh;
            if (st > pub_t) {
                if (lane == 0) atomicMax(&sc.ctrl->thresh, bias(st));
                pub_t = st;
            }
            const int cm = *(volatile int*)&s_cmax;
            if (use_bmax && cm > pub_cmax) {
                if (lane == 0) atomicMax(&sc.bmax[b], bias(cm));
                pub_cmax = cm;
            }
            unsigned bv[8];
            if (use_bmax) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int x = i * 32 + lane;
                    bv[i] = x < (int)G ? ld_relaxed_gpu(&sc.bmax[x]) : 0u;
                }
            }
            int t = kmax(st, unbias(ld_relaxed_gpu(&sc.ctrl->thresh)));
            if (use_bmax) {
                int ns = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int x = unbias(bv[i]);
                    const bool p = x > t;
                    const unsigned bb = __ballot_sync(kFullMask, p);
                    if (p) s_sel[ns + __popc(bb & lanemask_lt())] = x;
                    ns += __popc(bb);
                }
                __syncwarp();
                if (ns >= k) {
                    int sv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int p = i * 32 + lane;
                        sv[i] = p < ns ? s_sel[p] : INT_MIN;
                    }
                    warp_sort_desc<8>(sv, lane);
                    t = kmax(t, warp_sorted_at<8>(sv, k - 1));
                }
                __syncwarp();
            }
            if (t > st && lane == 0) atomicMax(&s_thresh, t);
            if (*(volatile int*)&s_done == kCons) break;
            __nanosleep(256);
        }
    } else {
        // ---- consumers ----
        int* q = s_queue + warp * kQueue;
        int nq = 0;
        int t = INT_MIN;
        int pushed_max = INT_MIN;  // largest tile maximum this warp sent to s_cmax

        // Merge every full 32-chunk of the queue (with all_of_it, the rest
        // too) into the list; raise t to the list's k-th value.
        auto drain = [&](bool all_of_it) {
            while (nq >= 32 || (all_of_it && nq > 0)) {
                const int cnt = nq >= 32 ? 32 : nq;
                __syncwarp();
                const int c = lane < cnt ? q[nq - cnt + lane] : INT_MIN;
                __syncwarp();
                nq -= cnt;
                int one[1] = {c};
                warp_sort_desc<1>(one, lane);
                wl.merge_sorted32(one[0], cnt, lane);
            }
            if (wl.have >= k) {
                const int kth = warp_sorted_at<L>(wl.lst, k - 1);
                if (kth > t) {
                    t = kth;
                    if (lane == 0) atomicMax(&s_thresh, kth);
                }
            }
        };

        // Scalars outside the aligned body: at most 3 + 3, taken by consumer
        // warp 0 of block 0.
        if (b == 0 && warp == 0) {
            const size_t ns = sp.head + (n - sp.tail0);
            const size_t pos = (size_t)lane < sp.head ? (size_t)lane : sp.tail0 + (lane - sp.head);
            enqueue(q, nq, (size_t)lane < ns ? ordered<KIND>(in[pos]) : INT_MIN, INT_MIN, lane);
        }

        // The warp's i-th tile goes through stage i % kWarpStages; s_tile
        // holds the tile id of each stage's copy.
        int4* my_ring = ring + (size_t)warp * kWarpStages * kTileVec;
        uint64_t* my_bar = full_bar + warp * kWarpStages;
        int* my_tile = s_tile + warp * kWarpStages;
        const unsigned wp = (unsigned)b + (unsigned)G * (unsigned)warp;  // this warp's index p
        unsigned static_i = 0;   // static items used: R full rounds, then the piece
        int cur = nr > 0 ? (int)(((unsigned)b * kCons + (unsigned)warp) % (unsigned)nr) : 0;  // range claimed from
        bool done = false;       // no tile left anywhere
        bool waited = false;     // grid dependency waited for (the counters are the previous launch's until then)
        auto range_lo = [&](int c) -> unsigned { return (unsigned)((unsigned long long)D * (unsigned)c / (unsigned)nr); };
        // A claim in two steps, so that the atomic's round trip overlaps other
        // work: start_claim returns a static item, or -1, or (kCounter) says
        // that lane 0 holds a counter value in `got`; finish_claim turns that
        // into an item id, or -1 when every range is used up.
        constexpr int kCounter = -2;
        unsigned got = 0;
        auto start_claim = [&]() -> int {
            while (static_i < R) {
                const unsigned id = wp + P * static_i++;
                size_t bs;
                unsigned c;
                item_span(id, bs, c);
                if (c) return (int)id;
            }
            if (static_i == R) {
                ++static_i;
                if (pieces && (wp < piece_r || piece_q > 0)) return (int)(R * P + wp);
            }
            if (done || nr == 0) return -1;
            if (!waited) {
                grid_dependency_wait();
                waited = true;
            }
            if (lane == 0) got = atomicAdd(dyn_counter(sc, cur), 1u);
            return kCounter;
        };
        auto finish_claim = [&](int raw) -> int {
            if (raw != kCounter) return raw;
            for (int tries = 0; tries <= 2 * kI32DynRanges + 2; ++tries) {
                got = __shfl_sync(kFullMask, got, 0);
                const unsigned lo = range_lo(cur), len = range_lo(cur + 1) - lo;
                if (got < len) return (int)(dyn_id0 + lo + got);
                // Range `cur` is used up (for good: its counter only grows).
                // Read every counter once and move to the first range after
                // it, cyclically, that still has tiles.
                unsigned word[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = h * 32 + lane;
                    bool left = false;
                    if (c < nr) left = ld_relaxed_gpu(dyn_counter(sc, c)) < range_lo(c + 1) - range_lo(c);
                    word[h] = __ballot_sync(kFullMask, left);
                }
                const unsigned long long has = ((unsigned long long)word[1] << 32) | word[0];
                const unsigned long long after = cur < 63 ? has & (~0ull << (cur + 1)) : 0ull;
                const unsigned long long pickm = after ? after : has;
                if (pickm == 0ull) {
                    done = true;
                    return -1;
                }
                cur = __ffsll((long long)pickm) - 1;
                if (lane == 0) got = atomicAdd(dyn_counter(sc, cur), 1u);
            }
            // Not reachable: each failed try finds one more range used up.
            if (lane == 0) atomicOr(sc.status, kStatusWaitTimeout);
            done = true;
            return -1;
        };
        auto issue = [&](unsigned i, int tile) {  // whole warp; lane 0 copies
            const int st = (int)(i % kWarpStages);
            if (lane == 0) {
                my_tile[st] = tile;
                size_t base;
                unsigned cnt;
                item_span((unsigned)tile, base, cnt);
                mbar_arrive_expect_tx(&my_bar[st], (uint32_t)(cnt * 16));
                // Default L2 policy.  Evict-first keeps the kernel's code in
                // L2 for its cold end (ticket, second stage) across
                // back-to-back launches, but measured slower in the bench
                // (1e8, k = 20: 71.5 against 66.6 us per call in a stream,
                // 81.9 against 77.8 us alone after an L2 flush).
                bulk_copy_g2s(my_ring + (size_t)st * kTileVec, sp.body + base, (uint32_t)(cnt * 16), &my_bar[st]);
            }
            __syncwarp();
        };
        if (use_tmax && !waited) {  // tile maxima go to the scratch
            grid_dependency_wait();
            waited = true;
        }

        unsigned issued = 0;
        while (issued < (unsigned)kWarpStages) {
            const int t = finish_claim(start_claim());
            if (t < 0) break;
            issue(issued++, t);
        }
        int pending = issued == (unsigned)kWarpStages ? start_claim() : -1;

        bool first = true;
        unsigned i = 0;
        for (; i < issued; ++i) {
            const int stg = (int)(i % kWarpStages);
            if (!mbar_wait(&my_bar[stg], (uint32_t)((i / kWarpStages) & 1))) {
                if (lane == 0) atomicOr(sc.status, kStatusWaitTimeout);
                // A claim in progress must not be lost: finish it and give
                // its tile to nobody (the status word marks the result bad).
                finish_claim(pending);
                pending = -1;
                break;
            }
            const unsigned tile = (unsigned)my_tile[stg];
            size_t base;
            unsigned cnt;
            item_span(tile, base, cnt);
            const int4* st = my_ring + (size_t)stg * kTileVec;
            int4 r[kU];
            if (cnt == (unsigned)kTileVec) {
#pragma unroll
                for (int u = 0; u < kU; ++u) r[u] = st[u * 32 + lane];
#pragma unroll
                for (int u = 0; u < kU; ++u) r[u] = ordered4<KIND>(r[u]);
            } else {
#pragma unroll
                for (int u = 0; u < kU; ++u)
                    r[u] = (unsigned)(u * 32 + lane) < cnt ? ordered4<KIND>(st[u * 32 + lane])
                                                         : make_int4(INT_MIN, INT_MIN, INT_MIN, INT_MIN);
            }
            __syncwarp();
            // The tile is in registers: re-arm its stage with the next tile
            // (claimed one tile earlier), and start the claim after that.
            {
                const int t = finish_claim(pending);
                pending = -1;
                if (t >= 0) {
                    if (lane == 0) fence_proxy_async_smem();
                    issue(issued++, t);
                    pending = start_claim();
                }
            }

            if (first) {
                // Start value: k-th largest of the tile's 32*GL group maxima.
                first = false;
                const int seed = seed_from_groups<GL>(r, k, lane);
                if (seed > t) {
                    t = seed;
                    if (lane == 0) atomicMax(&s_thresh, seed);
                }
            }
            t = kmax(t, *(volatile int*)&s_thresh);

            int m = INT_MIN;
#pragma unroll
            for (int u = 0; u < kU; ++u) m = kmax(m, max4(r[u]));
            const int wm = __reduce_max_sync(kFullMask, m);
            if (use_tmax && lane == 0) sc.tmax[tile] = wm;
            if (wm > pushed_max) {
                if (lane == 0) atomicMax(&s_cmax, wm);
                pushed_max = wm;
            }
            if (wm > t) {
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    if (__any_sync(kFullMask, max4(r[u]) > t)) {
                        enqueue(q, nq, r[u].x, t, lane);
                        enqueue(q, nq, r[u].y, t, lane);
                        enqueue(q, nq, r[u].z, t, lane);
                        enqueue(q, nq, r[u].w, t, lane);
                        if (nq >= 32) drain(false);
                    }
                }
            }
        }

        // After an early exit, let the copies this warp issued land before
        // the block moves on.
        for (unsigned w2 = i + 1; w2 < issued; ++w2)
            if (!mbar_wait(&my_bar[w2 % kWarpStages], (uint32_t)((w2 / kWarpStages) & 1))) break;
        drain(true);
        if (lane == 0) atomicAdd(&s_done, 1);
    }

    // Everything below uses the scratch: the previous launch must be done.
    grid_dependency_wait();

    // Block combine (section 2.1's tree, with warps in place of threads):
    // three levels of pairwise bitonic merges of the consumers' register
    // lists through shared memory.
    if (warp < kCons) {
#pragma unroll
        for (int i = 0; i < L; ++i) s_queue[warp * kQueue + i * 32 + lane] = wl.lst[i];
    }
    __syncthreads();
#pragma unroll
    for (int step = 1; step < kCons; step <<= 1) {
        if (warp < kCons && (warp & (2 * step - 1)) == 0 && warp + step < kCons) {
            const int* o = s_queue + (warp + step) * kQueue;
            // The other list reversed against ours: the half-cleaner of a
            // bitonic merge, then the merge network.
#pragma unroll
            for (int i = 0; i < L; ++i) wl.lst[i] = kmax(wl.lst[i], o[K - 1 - (i * 32 + lane)]);
            wl.bitonic_merge(lane);
#pragma unroll
            for (int i = 0; i < L; ++i) s_queue[warp * kQueue + i * 32 + lane] = wl.lst[i];
        }
        __syncthreads();
    }
    // The block's list, and how many of its entries exceed the grid
    // threshold now (only those can matter).
    if (threadIdx.x == 0) s_count = kmax(s_thresh, unbias(ld_relaxed_gpu(&sc.ctrl->thresh)));
    __syncthreads();
    const int t_now = s_count;
    if (warp == 0) write_list<L>(sc, (int)b, wl.lst, t_now, lane);
    const int block_kth = s_queue[k - 1];

    // This block has read all its input: the next launch on the stream may
    // start its blocks (they wait for this grid before touching the scratch),
    // when the caller keeps track of what this launch writes.
    if (release) launch_dependents();
    // Every threshold this block's warps used went through s_thresh: publish
    // it (and the block's k-th value) before the ticket, whatever the
    // monitor managed to do.
    if (block_done(sc, kmax(s_thresh, block_kth), &s_last))
        second_stage<KIND>(sc, k, 1, K, out, reinterpret_cast<int*>(ring), kRingBytes / (int)sizeof(int), cap_limit,
                     &s_count, use_tmax ? (int)sp.ntiles : 0);
}

// ------------------------------------------------------------ host side --

template <int L, int GL, int KIND>
struct StreamVariant {
    static constexpr int kThreads = kStreamThreads;
    static size_t smem_bytes() { return kRingBytes; }
    static const void* fn() { return reinterpret_cast<const void*>(&topk_i32_stream_kernel<L, GL, KIND>); }
    // Launched with programmatic stream serialization: when the previous
    // kernel on the stream is one of these, this one's blocks start once all
    // of that kernel's blocks have read their input, and overlap its last
    // block's second stage; every access to the shared scratch waits for it.
    static cudaError_t launch(int grid, cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out,
                              unsigned char* scratch, int cap_limit, bool early, bool release, int static_pct) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem_bytes();
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = early ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, topk_i32_stream_kernel<L, GL, KIND>, in, n, k, out, scratch, cap_limit,
                                  release ? 1 : 0, static_pct);
    }
    static size_t units_per_block() { return kCons; }
};

template <int KIND>
using VarK32 = StreamVariant<1, 1, KIND>;
template <int KIND>
using VarK64 = StreamVariant<2, 2, KIND>;
template <int KIND>
using VarK128 = StreamVariant<4, 4, KIND>;

// Blocks per SM and SM count of a kernel variant on a device, found once
// (the shared-memory opt-in is set at the same time) and cached.
struct DeviceFit {
    int sms = 0;
    int per_sm = 0;
};

template <class V>
cudaError_t device_fit(int device, DeviceFit* out) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static DeviceFit cache[kMaxDev];
    if (device < 0 || device >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[device].sms == 0) {
        DeviceFit f;
        cudaError_t e = cudaDeviceGetAttribute(&f.sms, cudaDevAttrMultiProcessorCount, device);
        if (e != cudaSuccess) return e;
        const size_t smem = V::smem_bytes();
        if (smem > 48 * 1024) {
            e = cudaFuncSetAttribute(V::fn(), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&f.per_sm, V::fn(), V::kThreads, smem);
        if (e != cudaSuccess) return e;
        if (f.per_sm < 1) f.per_sm = 1;
        cache[device] = f;
    }
    *out = cache[device];
    return cudaSuccess;
}

template <class V>
cudaError_t plan_for(int device, size_t n, I32Plan* plan) {
    DeviceFit f;
    cudaError_t e = device_fit<V>(device, &f);
    if (e != cudaSuccess) return e;
    size_t full = (size_t)f.sms * f.per_sm;
    if (full > (size_t)kI32MaxGrid) full = kI32MaxGrid;
    const size_t nvec = n / 4;
    const size_t tiles = (nvec + kTileVec - 1) / kTileVec;
    const size_t want = (tiles + V::units_per_block() - 1) / V::units_per_block();
    size_t grid = full;
    if (want < grid) grid = want;
    if (grid < 1) grid = 1;
    plan->grid = (int)grid;
    plan->max_grid = (int)full;
    plan->stage2_cap = stage2_cap_option();
    const int opt = stream_static_option();
    plan->static_pct = opt > 0 ? opt - 1 : kStaticPct;
    return cudaSuccess;
}

}  // namespace

namespace {

template <int KIND>
cudaError_t plan_kind(int device, size_t n, int k, I32Plan* plan) {
    if (k <= 32) return plan_for<VarK32<KIND>>(device, n, plan);
    if (k <= 64) return plan_for<VarK64<KIND>>(device, n, plan);
    return plan_for<VarK128<KIND>>(device, n, plan);
}

template <int KIND>
cudaError_t launch_kind(const I32Plan& plan, cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out,
                        unsigned char* sc, bool early, bool release) {
    const int cap = plan.stage2_cap, sp = plan.static_pct;
    if (k <= 32) return VarK32<KIND>::launch(plan.grid, s, in, n, k, out, sc, cap, early, release, sp);
    if (k <= 64) return VarK64<KIND>::launch(plan.grid, s, in, n, k, out, sc, cap, early, release, sp);
    return VarK128<KIND>::launch(plan.grid, s, in, n, k, out, sc, cap, early, release, sp);
}

}  // namespace

cudaError_t i32_plan(int device, size_t n, int k, I32Plan* plan, int kind) {
    plan->kind = kind;
    if (kind == kKeyU32) return plan_kind<kKeyU32>(device, n, k, plan);
    if (kind == kKeyF32) return plan_kind<kKeyF32>(device, n, k, plan);
    return plan_kind<kKeyI32>(device, n, k, plan);
}

cudaError_t i32_launch(const I32Plan& plan, cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out,
                       void* scratch, bool early, bool release) {
    auto* sc = static_cast<unsigned char*>(scratch);
    if (plan.kind == kKeyU32) return launch_kind<kKeyU32>(plan, s, in, n, k, out, sc, early, release);
    if (plan.kind == kKeyF32) return launch_kind<kKeyF32>(plan, s, in, n, k, out, sc, early, release);
    return launch_kind<kKeyI32>(plan, s, in, n, k, out, sc, early, release);
}

}  // namespace topk
