// Warp- and block-level building blocks shared by the TopK kernels.
//
// The pages' kernel ("CUDA parallel optimisation: TopK, shared memory and
// two-stage reduction", section 2.1) keeps one insertion-sorted list per
// thread and merges the lists pairwise through shared memory.  Here the lists
// are per warp, and sorting/merging is done with bitonic networks: across
// lanes with __shfl_xor_sync (the warp-shuffle reduction of "Complete guide
// to CUDA reduction optimisation", warp-shuffle section), and across
// registers or shared memory for wider lists.
#pragma once

#include <climits>
#include <cstdint>

namespace topk {

constexpr unsigned kFullMask = 0xffffffffu;

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ int kmax(int a, int b) { return a > b ? a : b; }
__device__ __forceinline__ int kmin(int a, int b) { return a < b ? a : b; }
__device__ __forceinline__ unsigned kmax(unsigned a, unsigned b) { return a > b ? a : b; }
__device__ __forceinline__ unsigned kmin(unsigned a, unsigned b) { return a < b ? a : b; }
__device__ __forceinline__ unsigned long long kmax(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}
__device__ __forceinline__ unsigned long long kmin(unsigned long long a, unsigned long long b) {
    return a < b ? a : b;
}

// Bitonic sort, descending, of the 32*N keys a warp holds in registers.
// Key j of lane l sits at position p = j*32 + l.  Strides below 32 exchange
// across lanes (shuffle); strides of 32 and more exchange between registers
// of the same lane.  After the call position 0 holds the largest key.
template <int N, typename T>
__device__ __forceinline__ void warp_sort_desc(T (&v)[N], int lane) {
#pragma unroll
    for (int size = 2; size <= 32 * N; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= 32) {
                const int js = stride >> 5;
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    if ((j & js) == 0) {
                        const int p = j * 32 + lane;
                        const bool desc = (p & size) == 0;
                        const T a = v[j], b = v[j | js];
                        const bool swap = desc ? (a < b) : (a > b);
                        v[j] = swap ? b : a;
                        v[j | js] = swap ? a : b;
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    const int p = j * 32 + lane;
                    const T other = __shfl_xor_sync(kFullMask, v[j], stride);
                    const bool lower = (lane & stride) == 0;
                    const bool desc = (p & size) == 0;
                    v[j] = (lower == desc) ? kmax(v[j], other) : kmin(v[j], other);
                }
            }
        }
    }
}

// The key at sorted position `pos` (0 <= pos < 32*N) of a warp_sort_desc
// result, returned to every lane.
template <int N, typename T>
__device__ __forceinline__ T warp_sorted_at(const T (&v)[N], int pos) {
    T mine = v[0];
#pragma unroll
    for (int j = 1; j < N; ++j)
        if (j == (pos >> 5)) mine = v[j];
    return __shfl_sync(kFullMask, mine, pos & 31);
}

// Bitonic sort, descending, of a[0..L) in shared memory by one warp.
// L is a power of two >= 2.
template <typename T>
__device__ void warp_sort_smem_desc(T* a, int L, int lane) {
    for (int size = 2; size <= L; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = lane; i < (L >> 1); i += 32) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const T x = a[lo], y = a[hi];
                if (desc ? (x < y) : (x > y)) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
            __syncwarp();
        }
    }
}

// Bitonic merge, descending, of a bitonic sequence a[0..L) in shared memory
// by one warp.  L is a power of two.
template <typename T>
__device__ void warp_merge_smem_desc(T* a, int L, int lane) {
    for (int stride = L >> 1; stride > 0; stride >>= 1) {
        for (int i = lane; i < (L >> 1); i += 32) {
            const int lo = 2 * i - (i & (stride - 1));
            const int hi = lo + stride;
            const T x = a[lo], y = a[hi];
            if (x < y) {
                a[lo] = y;
                a[hi] = x;
            }
        }
        __syncwarp();
    }
}

// Bitonic sort, descending, of a[0..L) in shared memory by the whole block.
// Every thread of the block must call it.  L is a power of two >= 2.
template <typename T>
__device__ void block_sort_smem_desc(T* a, int L) {
    __syncthreads();
    for (int size = 2; size <= L; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < (L >> 1); i += blockDim.x) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const T x = a[lo], y = a[hi];
                if (desc ? (x < y) : (x > y)) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
            __syncthreads();
        }
    }
}

__host__ __device__ __forceinline__ int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

}  // namespace topk
