// Score-keyed TopK with item ids, with an optional filter in front
// ("CUDA parallel optimisation: TopK, shared memory and two-stage
// reduction", section 6: update_candidates(candidates, k, item, score); its
// closing remark on composing stages -- filter first, then TopK; merge
// several TopK results).
//
// Among the positions i with keep[i] != 0 (every position when keep is
// null), the k best by score -- value descending, NaN above +inf, -0 equal
// to +0, the lower position first among equal scores -- with their scores
// (the input bits) and items (item[i], or i when item is null).
//
// Plan: the page's two-stage reduction, applied level by level with the row
// kernel (topk_rows.cu) as the block-level TopK:
//   filter   (keep given, large n, k <= 128) folded into level 1: the row
//            kernel skips filtered elements and says how many winners each
//            row has; a gather packs the rows' winners and the kept tail in
//            position order, padding at the end.  Otherwise an ordered
//            compaction of the kept scores and their positions (per-block
//            counts over contiguous ranges, then every block writes its kept
//            elements at its offset, in order) comes first.
//   level 1  the m candidates, as rows of C >= 8k scores plus one shorter
//            tail row: the row kernel leaves each row's k best.
//   level j  the previous level's winners, in row order, are the next
//            level's candidates.  Equal scores stay in position order: rows
//            are in position order, and a row's winners with equal scores
//            come in column order.  For k <= 128 a level is a chunk round
//            (each block keeps the k best of 1024 candidates, in order);
//            larger k take row-kernel levels.  Repeat until at most
//            kFinalCap candidates are left.
//   final    one block ranks those; the best k map back to input positions,
//            items and score bits.
// Merging several TopK results is this call on their concatenation.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "../../include/topk.h"
#include "topk_device.cuh"
#include "topk_internal.h"

namespace topk {

namespace {

constexpr int kFiltThreads = 512;
constexpr int kFiltMaxGrid = 1024;

// Per-block counts of kept positions over contiguous ranges.
__global__ void __launch_bounds__(kFiltThreads)
items_count_kernel(const uint8_t* __restrict__ keep, size_t n, size_t per, unsigned* __restrict__ counts) {
    const size_t lo = (size_t)blockIdx.x * per, hi = lo + per < n ? lo + per : n;
    unsigned c = 0;
    for (size_t i = lo + threadIdx.x; i < hi; i += blockDim.x) c += keep[i] != 0;
    c = __reduce_add_sync(kFullMask, c);
    __shared__ unsigned s[kFiltThreads / 32];
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned t = 0;
        for (int w = 0; w < kFiltThreads / 32; ++w) t += s[w];
        counts[blockIdx.x] = t;
    }
}

// Nonzero bytes of a 32-bit word.
__device__ __forceinline__ unsigned nonzero_bytes(unsigned w) {
    return (unsigned)__popc((((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w) & 0x80808080u);
}

// Vector form of the two filter kernels, for 16-byte-aligned score and keep
// arrays and ranges of whole 16-element groups: thread t of a chunk takes
// the 16 consecutive elements of group t (one 16-byte keep load, four
// 16-byte score loads), kVecChunks chunks of loads in flight.
constexpr int kVecGroup = 16;
constexpr int kStageBytes = kFiltThreads * kVecGroup * 8;  // one chunk's kept scores and positions

__global__ void __launch_bounds__(kFiltThreads)
items_count_vec_kernel(const uint8_t* __restrict__ keep, size_t n, size_t per, unsigned* __restrict__ counts) {
    const size_t lo = (size_t)blockIdx.x * per, hi = lo + per < n ? lo + per : n;
    const uint4* kv = reinterpret_cast<const uint4*>(keep);
    unsigned c = 0;
    constexpr int kIn = 4;
    for (size_t g0 = lo / kVecGroup + threadIdx.x; g0 * kVecGroup < hi; g0 += (size_t)kIn * blockDim.x) {
        uint4 v[kIn];
#pragma unroll
        for (int u = 0; u < kIn; ++u) {
            const size_t g = g0 + (size_t)u * blockDim.x;
            v[u] = g * kVecGroup < hi ? __ldg(kv + g) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kIn; ++u)
            c += nonzero_bytes(v[u].x) + nonzero_bytes(v[u].y) + nonzero_bytes(v[u].z) + nonzero_bytes(v[u].w);
    }
    c = __reduce_add_sync(kFullMask, c);
    __shared__ unsigned s[kFiltThreads / 32];
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned t = 0;
        for (int w = 0; w < kFiltThreads / 32; ++w) t += s[w];
        counts[blockIdx.x] = t;
    }
}

// Ordered compaction: block b writes its kept (score, position) pairs at the
// sum of the counts of the blocks before it, chunk by chunk in position
// order.  Block 0 also writes the total.
__global__ void __launch_bounds__(kFiltThreads)
items_compact_kernel(const float* __restrict__ score, const uint8_t* __restrict__ keep, size_t n, size_t per,
                     const unsigned* __restrict__ counts, float* __restrict__ cs, int32_t* __restrict__ cpos,
                     unsigned* __restrict__ total) {
    __shared__ unsigned s_warp[kFiltThreads / 32];
    __shared__ unsigned s_before[kFiltThreads / 32], s_all[kFiltThreads / 32];
    __shared__ unsigned s_base;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    // This block's offset (counts of the blocks before it) and, for block 0,
    // the total: a block-wide sum over at most kFiltMaxGrid counts.
    {
        unsigned before = 0, all = 0;
        for (unsigned j = threadIdx.x; j < gridDim.x; j += blockDim.x) {
            const unsigned c = counts[j];
            before += j < blockIdx.x ? c : 0u;
            all += c;
        }
        before = __reduce_add_sync(kFullMask, before);
        all = __reduce_add_sync(kFullMask, all);
        if (lane == 0) {
            s_before[w] = before;
            s_all[w] = all;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned b = 0, t = 0;
            for (int j = 0; j < kFiltThreads / 32; ++j) {
                b += s_before[j];
                t += s_all[j];
            }
            s_base = b;
            if (blockIdx.x == 0) *total = t;
        }
    }
    __syncthreads();
    unsigned base = s_base;
    const size_t lo = (size_t)blockIdx.x * per, hi = lo + per < n ? lo + per : n;
    for (size_t c0 = lo; c0 < hi; c0 += blockDim.x) {
        const size_t i = c0 + threadIdx.x;
        const bool p = i < hi && keep[i] != 0;
        const unsigned b = __ballot_sync(kFullMask, p);
        if (lane == 0) s_warp[w] = __popc(b);
        __syncthreads();
        unsigned before = 0, all = 0;
        for (int j = 0; j < kFiltThreads / 32; ++j) {
            const unsigned v = s_warp[j];
            before += j < w ? v : 0u;
            all += v;
        }
        if (p) {
            const unsigned slot = base + before + __popc(b & lanemask_lt());
            cs[slot] = score[i];
            cpos[slot] = (int32_t)i;
        }
        base += all;
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kFiltThreads)
items_compact_vec_kernel(const float* __restrict__ score, const uint8_t* __restrict__ keep, size_t n, size_t per,
                         const unsigned* __restrict__ counts, float* __restrict__ cs, int32_t* __restrict__ cpos,
                         unsigned* __restrict__ total) {
    extern __shared__ __align__(16) unsigned char items_stage_smem[];
    float* st_s = reinterpret_cast<float*>(items_stage_smem);                                  // one chunk's kept scores
    int32_t* st_p = reinterpret_cast<int32_t*>(items_stage_smem + kFiltThreads * kVecGroup * 4);  // and positions
    __shared__ unsigned s_warp[kFiltThreads / 32];
    __shared__ unsigned s_before[kFiltThreads / 32], s_all[kFiltThreads / 32];
    __shared__ unsigned s_base;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    {
        unsigned before = 0, all = 0;
        for (unsigned j = threadIdx.x; j < gridDim.x; j += blockDim.x) {
            const unsigned c = counts[j];
            before += j < blockIdx.x ? c : 0u;
            all += c;
        }
        before = __reduce_add_sync(kFullMask, before);
        all = __reduce_add_sync(kFullMask, all);
        if (lane == 0) {
            s_before[w] = before;
            s_all[w] = all;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned b = 0, t = 0;
            for (int j = 0; j < kFiltThreads / 32; ++j) {
                b += s_before[j];
                t += s_all[j];
            }
            s_base = b;
            if (blockIdx.x == 0) *total = t;
        }
    }
    __syncthreads();
    unsigned base = s_base;
    const size_t lo = (size_t)blockIdx.x * per, hi = lo + per < n ? lo + per : n;
    const uint4* kv = reinterpret_cast<const uint4*>(keep);
    const float4* sv = reinterpret_cast<const float4*>(score);
    for (size_t c0 = lo; c0 < hi; c0 += (size_t)blockDim.x * kVecGroup) {
        const size_t g = c0 / kVecGroup + threadIdx.x;  // this thread's group
        const bool in = g * kVecGroup < hi;
        const uint4 kb = in ? __ldg(kv + g) : make_uint4(0u, 0u, 0u, 0u);
        const unsigned words[4] = {kb.x, kb.y, kb.z, kb.w};
        unsigned mine = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) mine += nonzero_bytes(words[q]);
        // exclusive prefix of `mine` over the block (thread order = position order)
        unsigned x = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(kFullMask, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp[w] = x;
        __syncthreads();
        unsigned before = 0, all = 0;
        for (int j = 0; j < kFiltThreads / 32; ++j) {
            const unsigned v = s_warp[j];
            before += j < w ? v : 0u;
            all += v;
        }
        // This chunk's kept elements go to shared memory in position order,
        // then out to the compacted arrays with coalesced stores.
        unsigned slot = before + x - mine;
        if (mine) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 f = __ldg(sv + g * 4 + q);
                const float fs[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    if ((words[q] >> (8 * b)) & 0xFFu) {
                        st_s[slot] = fs[b];
                        st_p[slot] = (int32_t)(g * kVecGroup + q * 4 + b);
                        ++slot;
                    }
                }
            }
        }
        __syncthreads();
        for (unsigned i = threadIdx.x; i < all; i += blockDim.x) {
            cs[base + i] = st_s[i];
            cpos[base + i] = st_p[i];
        }
        base += all;
        __syncthreads();
    }
}

// Next level's candidates: this level's winners of its R full rows (R x ke,
// row r's columns counting from r * C), then the tail the rows did not cover
// (its candidates carried over as they are), then -inf pads up to `len`.
// Positions map through pos (null: identity).  Pads only ever sit at the end
// of an array, after every real candidate, so under the position tie-break
// they never beat a real one, not even a real -inf.
__global__ void items_gather_kernel(const float* __restrict__ wv, const int32_t* __restrict__ wx, int R, int C,
                                    int ke, const float* __restrict__ cur, const int32_t* __restrict__ pos,
                                    size_t tail_begin, size_t tail_len, size_t len, float* __restrict__ ns,
                                    int32_t* __restrict__ npos) {
    grid_dependency_wait();  // launched early (launch_pdl): the previous kernel's writes first
    launch_dependents();
    const size_t nw = (size_t)R * ke;
    for (size_t j = (size_t)blockIdx.x * blockDim.x + threadIdx.x; j < len; j += (size_t)gridDim.x * blockDim.x) {
        float v;
        int32_t p;
        if (j < nw) {
            const size_t src = (j / ke) * C + wx[j];
            v = wv[j];
            p = pos ? pos[src] : (int32_t)src;
        } else if (j < nw + tail_len) {
            const size_t src = tail_begin + (j - nw);
            v = cur[src];
            p = pos ? pos[src] : (int32_t)src;
        } else {
            v = __int_as_float(0xFF800000);  // -inf
            p = -1;
        }
        ns[j] = v;
        npos[j] = p;
    }
}

// Next level's candidates after a filtered level 1: the valid winners of
// the R rows (wc[r] of them in row r, first in its k outputs; row r's
// columns count from r * C), then the kept elements of the tail [R * C, n),
// all in position order, then (-inf, -1) pads up to `len`.  Block b packs
// rows [b * rb, (b + 1) * rb); the last block also packs the tail.
constexpr int kGatherThreads = 512;
__global__ void __launch_bounds__(kGatherThreads)
items_gather_masked_kernel(const float* __restrict__ wv, const int32_t* __restrict__ wx,
                           const int32_t* __restrict__ wc, int R, int C, int k, const float* __restrict__ score,
                           const uint8_t* __restrict__ keep, size_t n, size_t len, float* __restrict__ ns,
                           int32_t* __restrict__ npos) {
    __shared__ unsigned s_red[kGatherThreads / 32][2];
    __shared__ unsigned s_rowbase[kGatherThreads];
    __shared__ unsigned s_warp[kGatherThreads / 32];
    grid_dependency_wait();  // launched early (launch_pdl): the previous kernel's writes first
    launch_dependents();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int rb = (R + (int)gridDim.x - 1) / (int)gridDim.x;
    const int r0 = (int)blockIdx.x * rb < R ? (int)blockIdx.x * rb : R;
    const int r1 = r0 + rb < R ? r0 + rb : R;
    // Winners of the rows before this block's, and of all rows.
    unsigned before = 0, all = 0;
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        const unsigned c = (unsigned)wc[r];
        before += r < r0 ? c : 0u;
        all += c;
    }
    before = __reduce_add_sync(kFullMask, before);
    all = __reduce_add_sync(kFullMask, all);
    if (lane == 0) {
        s_red[w][0] = before;
        s_red[w][1] = all;
    }
    __syncthreads();
    before = all = 0;
    for (int j = 0; j < kGatherThreads / 32; ++j) {
        before += s_red[j][0];
        all += s_red[j][1];
    }
    // This block's rows, rb <= blockDim at a time: an exclusive scan of
    // their counts, then one warp per row copies its winners.
    for (int c0 = r0; c0 < r1; c0 += blockDim.x) {
        const int r = c0 + (int)threadIdx.x;
        const unsigned c = r < r1 ? (unsigned)wc[r] : 0u;
        unsigned x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(kFullMask, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp[w] = x;
        __syncthreads();
        unsigned wb = 0, tot = 0;
        for (int j = 0; j < kGatherThreads / 32; ++j) {
            wb += j < w ? s_warp[j] : 0u;
            tot += s_warp[j];
        }
        s_rowbase[threadIdx.x] = before + wb + x - c;
        __syncthreads();
        const int nr = r1 - c0 < (int)blockDim.x ? r1 - c0 : (int)blockDim.x;
        for (int i = w; i < nr; i += kGatherThreads / 32) {
            const int rr = c0 + i;
            const int cnt = wc[rr];
            const size_t dst = s_rowbase[i];
            for (int j = lane; j < cnt; j += 32) {
                ns[dst + j] = wv[(size_t)rr * k + j];
                npos[dst + j] = (int32_t)((size_t)rr * C + (size_t)wx[(size_t)rr * k + j]);
            }
        }
        before += tot;
        __syncthreads();
    }
    // Pads after the tail's room, by every block; the tail itself and the
    // pads in the rest of its room, by the last block.
    const size_t tail0 = (size_t)R * (size_t)C, tail_len = n - tail0;
    for (size_t j = all + tail_len + (size_t)blockIdx.x * blockDim.x + threadIdx.x; j < len;
         j += (size_t)gridDim.x * blockDim.x) {
        ns[j] = __int_as_float(0xFF800000);
        npos[j] = -1;
    }
    if (blockIdx.x != gridDim.x - 1) return;
    unsigned base = all;
    for (size_t c0 = tail0; c0 < n; c0 += blockDim.x) {
        const size_t i = c0 + threadIdx.x;
        const bool p = i < n && keep[i] != 0;
        const unsigned b = __ballot_sync(kFullMask, p);
        if (lane == 0) s_warp[w] = __popc(b);
        __syncthreads();
        unsigned wb = 0, tot = 0;
        for (int j = 0; j < kGatherThreads / 32; ++j) {
            wb += j < w ? s_warp[j] : 0u;
            tot += s_warp[j];
        }
        if (p) {
            const unsigned slot = base + wb + __popc(b & lanemask_lt());
            ns[slot] = score[i];
            npos[slot] = (int32_t)i;
        }
        base += tot;
        __syncthreads();
    }
    for (size_t j = base + threadIdx.x; j < all + tail_len && j < len; j += blockDim.x) {
        ns[j] = __int_as_float(0xFF800000);
        npos[j] = -1;
    }
}

// Order key of a score: value descending with NaN on top and -0 equal to +0
// (the row order), then the lower array index first.
__device__ __forceinline__ unsigned long long items_key(float v, unsigned j) {
    const unsigned b = __float_as_uint(v);
    unsigned k;
    if ((b & 0x7FFFFFFFu) > 0x7F800000u)
        k = 0xFFFFFFFFu;  // NaN
    else if ((b & 0x7FFFFFFFu) == 0u)
        k = 0x80000000u;  // +-0
    else
        k = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)k << 32) | (0xFFFFFFFFu - j);
}

// The last level: at most kFinalCap candidates (their array order is their
// position order among equal scores) sorted in one block; the best ke map
// to items and score bits, the rest of the k outputs are padding.
constexpr int kFinalCap = 4096;
constexpr int kFinalThreads = 1024;
__global__ void __launch_bounds__(kFinalThreads)
items_final_sort_kernel(const float* __restrict__ cv, const int32_t* __restrict__ cp, int count, int ke, int k,
                        const int64_t* __restrict__ item, float* __restrict__ out_score,
                        int64_t* __restrict__ out_item, int64_t* __restrict__ out_count) {
    __shared__ unsigned long long keys[kFinalCap];
    grid_dependency_wait();  // launched early (launch_pdl): the previous kernel's writes first
    // The call's last kernel: its successor must not start before it ends.
    const int L = next_pow2(count < 2 ? 2 : count);
    for (int j = threadIdx.x; j < L; j += blockDim.x) keys[j] = j < count ? items_key(cv[j], (unsigned)j) : 0ull;
    block_sort_smem_desc(keys, L);
    // Pads (position -1) sort after every real candidate, so the valid
    // outputs come first; their number is the count.
    int valid = 0;
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
        const unsigned idx = 0xFFFFFFFFu - (unsigned)(keys[j] & 0xFFFFFFFFull);
        const int32_t p = (j < ke && j < count) ? (cp ? cp[idx] : (int32_t)idx) : -1;
        if (p >= 0) {
            out_score[j] = cv[idx];
            out_item[j] = item ? item[p] : (int64_t)p;
            ++valid;
        } else {
            out_score[j] = __int_as_float(0xFF800000);
            out_item[j] = -1;
        }
    }
    static_assert(TOPK_MAX_K_ROWS <= kFinalThreads, "one output per thread: the count is a thread count");
    valid = __syncthreads_count(valid);
    if (threadIdx.x == 0 && out_count) *out_count = valid;
}

// The last level for k <= 128: each of 32 warps sorts its 128 of the at
// most kFinalCap candidates in registers, and the warps' lists are merged
// pairwise (five levels) into warp 0, whose best k are the outputs.  Same
// keys and outputs as items_final_sort_kernel.
constexpr int kSelWarps = 32, kSelN = kFinalCap / (32 * kSelWarps);  // 4 keys per lane
__global__ void __launch_bounds__(kSelWarps * 32)
items_final_select_kernel(const float* __restrict__ cv, const int32_t* __restrict__ cp, int count, int ke, int k,
                          const int64_t* __restrict__ item, float* __restrict__ out_score,
                          int64_t* __restrict__ out_item, int64_t* __restrict__ out_count) {
    __shared__ unsigned long long s_l[kSelWarps][32 * kSelN];
    grid_dependency_wait();  // launched early (launch_pdl): the previous kernel's writes first
    // The call's last kernel: its successor must not start before it ends.
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    // Warps whose slots start at or past `count` hold no candidate; they
    // skip the sort, and no merge takes their (empty) lists.
    auto live = [&](int warp) { return warp * 32 * kSelN < count; };
    RegList<kSelN, unsigned long long> wl;
#pragma unroll
    for (int j = 0; j < kSelN; ++j) {
        const int p = w * 32 * kSelN + j * 32 + lane;
        wl.lst[j] = p < count ? items_key(cv[p], (unsigned)p) : 0ull;  // every real key is above 0
    }
    if (live(w)) warp_sort_desc<kSelN>(wl.lst, lane);
#pragma unroll 1
    for (int s = 1; s < kSelWarps; s <<= 1) {
        if ((w & (2 * s - 1)) == s && live(w))
#pragma unroll
            for (int j = 0; j < kSelN; ++j) s_l[w][j * 32 + lane] = wl.lst[j];
        __syncthreads();
        if ((w & (2 * s - 1)) == 0 && live(w + s)) wl.merge_list(s_l[w + s], lane);
        __syncthreads();
    }
    if (w != 0) return;
    int valid = 0;
#pragma unroll
    for (int j = 0; j < kSelN; ++j) {
        const int o = j * 32 + lane;
        const unsigned long long key = wl.lst[j];
        const unsigned idx = 0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull);
        const int32_t p = (o < ke && key != 0ull) ? (cp ? cp[idx] : (int32_t)idx) : -1;
        if (o < k) {
            if (p >= 0) {
                out_score[o] = cv[idx];
                out_item[o] = item ? item[p] : (int64_t)p;
            } else {
                out_score[o] = __int_as_float(0xFF800000);
                out_item[o] = -1;
            }
        }
        valid += __popc(__ballot_sync(kFullMask, o < k && p >= 0));
    }
    if (lane == 0 && out_count) *out_count = valid;
}

// Later levels for k <= 128: block b takes candidates [b * kChunk,
// (b + 1) * kChunk) -- kChunkWarps warps of 256 -- ranks them like the
// final select (register sort per warp, pairwise merges) and writes its best
// ke, in order, at b * ke of the next arrays (pads, -inf and -1, when the
// chunk has fewer).  Chunks are in array order, so equal scores stay in
// position order; pads only ever sit at the end of the array, hence in the
// last chunks, and stay at the end.  Small blocks spread a round over every
// SM (the work is about 10 instructions per candidate, in register sorts).
// Measured per call on 1e8 scores, k = 64: 129 us with 4 warps per block,
// 131 with 8, 134 with 2, and 140 with 32 (8192 candidates per block, so
// the first round had 32 blocks).
constexpr int kChunkN = 8;                                 // keys per lane
constexpr int kChunkWarps = 4;
constexpr int kChunk = kChunkWarps * 32 * kChunkN;         // 1024 candidates per block
__global__ void __launch_bounds__(kChunkWarps * 32)
items_select_chunks_kernel(const float* __restrict__ cv, const int32_t* __restrict__ cp, size_t count, int ke,
                           float* __restrict__ nv, int32_t* __restrict__ np) {
    __shared__ unsigned long long s_l[kChunkWarps][32 * kSelN];
    grid_dependency_wait();  // launched early (launch_pdl): the previous kernel's writes first
    launch_dependents();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const size_t base = (size_t)blockIdx.x * kChunk + (size_t)w * 32 * kChunkN;
    // The warp's 256 candidates as two sorted halves of 128 (the same
    // register sort as the final select), merged through its own slot.
    RegList<kSelN, unsigned long long> wl;  // the warp's best 32 * kSelN >= ke
#pragma unroll 1
    for (int h = 0; h < kChunkN / kSelN; ++h) {
        unsigned long long v[kSelN];
#pragma unroll
        for (int j = 0; j < kSelN; ++j) {
            const size_t p = base + (size_t)(h * kSelN + j) * 32 + lane;
            v[j] = p < count ? items_key(cv[p], (unsigned)p) : 0ull;  // every real key is above 0
        }
        warp_sort_desc<kSelN>(v, lane);
        if (h == 0) {
#pragma unroll
            for (int j = 0; j < kSelN; ++j) wl.lst[j] = v[j];
        } else {
#pragma unroll
            for (int j = 0; j < kSelN; ++j) s_l[w][j * 32 + lane] = v[j];
            __syncwarp();
            wl.merge_list(s_l[w], lane);
            __syncwarp();
        }
    }
#pragma unroll 1
    for (int s = 1; s < kChunkWarps; s <<= 1) {
        if ((w & (2 * s - 1)) == s)
#pragma unroll
            for (int j = 0; j < kSelN; ++j) s_l[w][j * 32 + lane] = wl.lst[j];
        __syncthreads();
        if ((w & (2 * s - 1)) == 0) wl.merge_list(s_l[w + s], lane);
        __syncthreads();
    }
    if (w != 0) return;
#pragma unroll
    for (int j = 0; j < kSelN; ++j) {
        const int o = j * 32 + lane;
        if (o < ke) {
            const unsigned long long key = wl.lst[j];
            const unsigned idx = 0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull);
            const size_t dst = (size_t)blockIdx.x * ke + o;
            nv[dst] = key ? cv[idx] : __int_as_float(0xFF800000);
            np[dst] = key ? (cp ? cp[idx] : (int32_t)idx) : -1;
        }
    }
}

// Pads the outputs when nothing is kept.
__global__ void items_empty_kernel(int k, float* __restrict__ out_score, int64_t* __restrict__ out_item,
                                   int64_t* __restrict__ out_count) {
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
        out_score[j] = __int_as_float(0xFF800000);
        out_item[j] = -1;
    }
    if (threadIdx.x == 0 && out_count) *out_count = 0;
}

// Rows of the first level aim at kTargetRows (one warp per row fills the
// GPU); later levels, whose candidates are few, at kLaterRows.  A row holds
// at least 8 ke candidates, so every level shrinks them at least eightfold.
constexpr size_t kTargetRows = 4096;
constexpr size_t kLaterRows = 256;
inline size_t level_cols(size_t count, int ke, bool first) {
    const size_t rows = first ? kTargetRows : kLaterRows;
    size_t c = (count + rows - 1) / rows;
    if (c < (size_t)8 * ke) c = (size_t)8 * ke;
    return c;
}

// Largest number of candidates a later level holds, padding included.
inline size_t next_cap(size_t n, int k) {
    return (kTargetRows + 1) * (size_t)k + 4 * (n / kTargetRows + 32 * (size_t)k + 2);
}

// The filter folds into level 1 for large inputs, k <= 128 and a keep array
// whose 4-byte words line up with the score array's 16-byte vectors.
constexpr size_t kFusedMinN = size_t(1) << 20;

}  // namespace

bool items_fused_filter(const float* score, const uint8_t* keep, size_t n, int k) {
    return keep && n >= kFusedMinN && k <= 128 && rows_mask_aligned(score, keep);
}

size_t items_scratch_bytes(size_t n, int k, bool compact) {
    size_t b = 0;
    if (compact) b += kFiltMaxGrid * 4 + 256 + n * 8 + 512;  // counts, total, compacted scores and positions
    const size_t winners = (kTargetRows + 1) * (size_t)k;
    b += winners * 8 + 2 * next_cap(n, k) * 8 + 6 * 256;      // winners, two candidate arrays
    b += (kTargetRows + 1) * 4 + 256;                          // winners per row (filtered level 1)
    return b;
}

namespace {
std::mutex g_items_mu;
bool g_items_ready[64];
}  // namespace

cudaError_t items_launch(cudaStream_t s, const float* score, const int64_t* item, const uint8_t* keep, size_t n,
                         int k, float* out_score, int64_t* out_item, int64_t* out_count, void* scratch,
                         size_t scratch_bytes, unsigned* status, int* launches) {
    *launches = 0;
    const bool fused = items_fused_filter(score, keep, n, k);
    if (scratch_bytes < items_scratch_bytes(n, k, keep != nullptr && !fused)) return cudaErrorInvalidValue;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_items_mu);
        if (!g_items_ready[device]) {
            e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&items_compact_vec_kernel),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytes);
            if (e != cudaSuccess) return e;
            g_items_ready[device] = true;
        }
    }
    auto* base = static_cast<unsigned char*>(scratch);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        void* p = base + off;
        off += (bytes + 255) / 256 * 256;
        return p;
    };

    const float* cur = score;
    const int32_t* cur_pos = nullptr;
    size_t m = n;
    if (keep && !fused) {
        const size_t per0 = (n + kFiltMaxGrid - 1) / kFiltMaxGrid;
        const size_t per = per0 < (size_t)kFiltThreads ? (size_t)kFiltThreads : (per0 + 511) / 512 * 512;
        const int grid = (int)((n + per - 1) / per);
        auto* counts = static_cast<unsigned*>(take(kFiltMaxGrid * 4));
        auto* total = static_cast<unsigned*>(take(4));
        auto* cs = static_cast<float*>(take(n * 4));
        auto* cp = static_cast<int32_t*>(take(n * 4));
        // The vector kernels need 16-byte-aligned arrays and ranges of whole
        // 16-element groups: per is a multiple of 512, and n a multiple of 16.
        const bool vec = ((reinterpret_cast<uintptr_t>(keep) | reinterpret_cast<uintptr_t>(score)) & 15u) == 0 &&
                         n % kVecGroup == 0;
        if (vec) {
            items_count_vec_kernel<<<grid, kFiltThreads, 0, s>>>(keep, n, per, counts);
            items_compact_vec_kernel<<<grid, kFiltThreads, kStageBytes, s>>>(score, keep, n, per, counts, cs, cp,
                                                                            total);
        } else {
            items_count_kernel<<<grid, kFiltThreads, 0, s>>>(keep, n, per, counts);
            items_compact_kernel<<<grid, kFiltThreads, 0, s>>>(score, keep, n, per, counts, cs, cp, total);
        }
        *launches += 2;
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        // The plan of the levels depends on how many are kept: read it.
        unsigned h = 0;
        e = cudaMemcpyAsync(&h, total, 4, cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return e;
        m = h;
        cur = cs;
        cur_pos = cp;
        if (m == 0) {
            items_empty_kernel<<<1, 256, 0, s>>>(k, out_score, out_item, out_count);
            *launches += 1;
            return cudaGetLastError();
        }
    }
    const int ke = m < (size_t)k ? (int)m : k;  // with a fused filter m is not known here: ke = k
    const size_t winners = (kTargetRows + 1) * (size_t)k;
    auto* wv = static_cast<float*>(take(winners * 4));
    auto* wx = static_cast<int32_t*>(take(winners * 4));
    const size_t cap = next_cap(n, k);
    float* nb_s[2] = {static_cast<float*>(take(cap * 4)), nullptr};
    int32_t* nb_p[2] = {static_cast<int32_t*>(take(cap * 4)), nullptr};
    nb_s[1] = static_cast<float*>(take(cap * 4));
    nb_p[1] = static_cast<int32_t*>(take(cap * 4));
    int flip = 0;
    size_t len = m;      // entries of cur, pads included
    size_t real = m;     // entries of cur that are not pads (an upper bound after level 1)
    bool first = true;
    if (fused) {
        // Level 1 over the kept elements of the whole input, then the packed
        // winners and kept tail (pads at the end) are the next candidates.
        auto* wc = static_cast<int32_t*>(take((kTargetRows + 1) * 4));
        // The last block of the gather packs the tail alone: keep it short.
        // Rows of n / kTargetRows leave fewer than kTargetRows elements over
        // whenever that is a row's worth of at least 8k; otherwise the
        // rounded-up rows are short themselves (fewer than kTargetRows).
        size_t C = n / kTargetRows;
        if (C < (size_t)8 * ke || C <= n % kTargetRows) C = level_cols(n, ke, true);
        const size_t R = n / C;
        // Every kernel from here on waits for its predecessor before it
        // reads anything, so each is launched early (programmatic stream
        // serialization) and only the launch gaps go.
        e = rows_launch_masked(s, score, keep, (int)R, (int)C, ke, wv, wx, wc, status, true,
                               kRowsRelease | kRowsWaitFirst);
        if (e != cudaSuccess) return e;
        *launches += 1;
        const size_t next_real = R * ke + (n - R * C);
        const size_t Cn = level_cols(next_real, ke, false);
        const size_t next_len = next_real <= (size_t)kFinalCap ? next_real : (next_real + Cn - 1) / Cn * Cn;
        const int gb = R < 128 ? (R < 1 ? 1 : (int)R) : 128;
        e = launch_pdl(items_gather_masked_kernel, gb, kGatherThreads, 0, s, wv, wx, wc, (int)R, (int)C, ke, score,
                       keep, n, next_len, nb_s[0], nb_p[0]);
        *launches += 1;
        if (e != cudaSuccess) return e;
        cur = nb_s[0];
        cur_pos = nb_p[0];
        flip = 1;
        len = next_len;
        real = next_real;
        first = false;
    }
    for (;;) {
        if (real <= (size_t)kFinalCap) {
            // cur holds real entries only here (a single-row level adds no pads)
            *launches += 1;
            if (k <= 32 * kSelN)
                return launch_pdl(items_final_select_kernel, 1, kSelWarps * 32, 0, s, cur, cur_pos, (int)real, ke, k,
                                  item, out_score, out_item, out_count);
            return launch_pdl(items_final_sort_kernel, 1, kFinalThreads, 0, s, cur, cur_pos, (int)real, ke, k, item,
                              out_score, out_item, out_count);
        }
        if (!first && k <= 32 * kSelN) {
            // A chunk round: ceil(len / kChunk) blocks each keep their ke best.
            const size_t nb = (len + kChunk - 1) / kChunk;
            e = launch_pdl(items_select_chunks_kernel, (unsigned)nb, kChunkWarps * 32, 0, s, cur, cur_pos, len, ke,
                           nb_s[flip], nb_p[flip]);
            *launches += 1;
            if (e != cudaSuccess) return e;
            cur = nb_s[flip];
            cur_pos = nb_p[flip];
            flip ^= 1;
            len = real = nb * (size_t)ke;
            continue;
        }
        size_t C = level_cols(real, ke, first);
        if (C > len) C = len;  // fewer candidates than one row of 8 ke: a single row of all of them
        const size_t R = len / C, tail = len - R * C;  // later levels: len is a multiple of C, tail 0
        e = rows_launch(s, cur, (int)R, (int)C, ke, wv, wx, status, true, kRowsRelease | kRowsWaitFirst);
        if (e != cudaSuccess) return e;
        *launches += 1;
        const size_t next_real = R * ke + tail;
        const size_t Cn = level_cols(next_real, ke, false);
        const size_t next_len = next_real <= (size_t)kFinalCap ? next_real : (next_real + Cn - 1) / Cn * Cn;
        const int gb = (int)((next_len + 255) / 256 < 1024 ? (next_len + 255) / 256 : 1024);
        e = launch_pdl(items_gather_kernel, gb, 256, 0, s, wv, wx, (int)R, (int)C, ke, cur, cur_pos, R * C, tail,
                       next_len, nb_s[flip], nb_p[flip]);
        *launches += 1;
        if (e != cudaSuccess) return e;
        cur = nb_s[flip];
        cur_pos = nb_p[flip];
        flip ^= 1;
        len = next_len;
        real = next_real;
        first = false;
    }
}

}  // namespace topk
