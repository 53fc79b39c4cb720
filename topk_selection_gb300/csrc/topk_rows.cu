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
    if constexpr (B == 256) {
        u64 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int p = j * 32 + lane;
            v[j] = p < w.cnt ? w.buf[p] : 0ull;
        }
        warp_sort_desc<8>(v, lane);
        const int keep = w.cnt < k ? w.cnt : k;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int p = j * 32 + lane;
            if (p < keep) w.buf[p] = v[j];
        }
        if (w.cnt >= k) {
            const u64 kth = warp_sorted_at<8>(v, k - 1);
            if (kth > w.T) {
                w.T = kth;
                raised = true;
            }
        }
        w.cnt = keep;
    } else {
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
    }
    __syncwarp();
    return raised;
}

template <int B>
__global__ void __launch_bounds__(kWarps * 32, (B <= 256 ? 4 : 1))
topk_rows_kernel(const float* __restrict__ in, int cols, int k, float* __restrict__ vals,
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

}  // namespace

cudaError_t rows_launch(cudaStream_t s, const float* in, int rows, int cols, int k, float* vals, int32_t* idx) {
    if (k <= 128) {
        const size_t smem = (size_t)kWarps * 256 * sizeof(u64);
        topk_rows_kernel<256><<<rows, kWarps * 32, smem, s>>>(in, cols, k, vals, idx);
    } else {
        const size_t smem = (size_t)kWarps * 2048 * sizeof(u64);
        cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&topk_rows_kernel<2048>),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        topk_rows_kernel<2048><<<rows, kWarps * 32, smem, s>>>(in, cols, k, vals, idx);
    }
    return cudaGetLastError();
}

}  // namespace topk
