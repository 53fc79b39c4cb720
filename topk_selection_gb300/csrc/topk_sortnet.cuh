// A block-wide bitonic sort that keeps most of its stages in registers.
//
// The plain shared-memory network (block_sort_smem_desc) spends a block
// barrier on every stage: 55 of them for 1024 keys.  Here warp w holds the
// 64 consecutive elements 64w + lane and 64w + 32 + lane in two registers,
// so strides below 32 are lane exchanges (__shfl_xor_sync, as in the
// warp-shuffle level of "Complete guide to CUDA reduction optimisation") and
// a stride of 32 is a register exchange; only strides of 64 and more go
// through shared memory, with two barriers each (10 such stages for 1024
// keys, 15 for 2048).
#pragma once

#include "topk_device.cuh"

namespace topk {

// Sort a[0, L) descending.  kThreads is the block size; L is a power of two
// with 64 <= L <= 2 * kThreads.  Every thread of the block must call it.
template <typename T, int kThreads>
__device__ void block_sort_reg_desc(T* a, int L) {
    static_assert(kThreads % 32 == 0, "whole warps");
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const bool act = 64 * w < L;  // L is a multiple of 64: an active warp's 64 elements are all in range
    const int e0 = 64 * w + lane, e1 = e0 + 32;
    T x0 = T(0), x1 = T(0);
    __syncthreads();
    if (act) {
        x0 = a[e0];
        x1 = a[e1];
    }
    // Strides `from` down to 1 of the merge for sequences of `size`.
    auto reg_stages = [&](int size, int from) {
        for (int st = from; st > 0; st >>= 1) {
            const bool d0 = (e0 & size) == 0, d1 = (e1 & size) == 0;  // descending here
            if (st == 32) {
                const T hi = kmax(x0, x1), lo = kmin(x0, x1);
                x0 = d0 ? hi : lo;
                x1 = d0 ? lo : hi;
            } else {
                const T y0 = __shfl_xor_sync(kFullMask, x0, st), y1 = __shfl_xor_sync(kFullMask, x1, st);
                const bool low = (lane & st) == 0;
                x0 = low == d0 ? kmax(x0, y0) : kmin(x0, y0);
                x1 = low == d1 ? kmax(x1, y1) : kmin(x1, y1);
            }
        }
    };
    if (act)
        for (int size = 2; size <= 64; size <<= 1) reg_stages(size, size >> 1);
    for (int size = 128; size <= L; size <<= 1) {
        for (int st = size >> 1; st >= 64; st >>= 1) {
            if (act) {
                a[e0] = x0;
                a[e1] = x1;
            }
            __syncthreads();
            if (act) {
                const T y0 = a[e0 ^ st], y1 = a[e1 ^ st];
                const bool d0 = (e0 & size) == 0, d1 = (e1 & size) == 0;
                x0 = ((e0 & st) == 0) == d0 ? kmax(x0, y0) : kmin(x0, y0);
                x1 = ((e1 & st) == 0) == d1 ? kmax(x1, y1) : kmin(x1, y1);
            }
            __syncthreads();
        }
        if (act) reg_stages(size, 32);
    }
    if (act) {
        a[e0] = x0;
        a[e1] = x1;
    }
    __syncthreads();
}

}  // namespace topk
