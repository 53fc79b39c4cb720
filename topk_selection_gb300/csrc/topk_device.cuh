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

#include "topk_internal.h"

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

// A warp's sorted (descending) top-K list of keys, K = 32*L, held in
// registers: position p = j*32 + lane is lst[j] of lane `lane`.
template <int L, typename T>
struct RegList {
    T lst[L];
    int have;  // real entries (the rest hold the sentinel)

    __device__ __forceinline__ void init(T sentinel) {
#pragma unroll
        for (int j = 0; j < L; ++j) lst[j] = sentinel;
        have = 0;
    }

    // Sort a bitonic list descending (the merge half of a bitonic sort).
    __device__ __forceinline__ void bitonic_merge(int lane) {
#pragma unroll
        for (int stride = 16 * L; stride > 0; stride >>= 1) {
            if (stride >= 32) {
                const int js = stride >> 5;
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    if ((j & js) == 0) {
                        const T a = lst[j], b = lst[j | js];
                        lst[j] = kmax(a, b);
                        lst[j | js] = kmin(a, b);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    const T o = __shfl_xor_sync(kFullMask, lst[j], stride);
                    lst[j] = (lane & stride) == 0 ? kmax(lst[j], o) : kmin(lst[j], o);
                }
            }
        }
    }

    // Merge a sorted-descending 32-chunk (one key per lane, position = lane)
    // into the list, keeping the K largest: the half-cleaner against the
    // reversed chunk, then the merge network.
    __device__ __forceinline__ void merge_sorted32(T c, int cnt, int lane) {
        const T rc = __shfl_sync(kFullMask, c, 31 - lane);
        lst[L - 1] = kmax(lst[L - 1], rc);
        bitonic_merge(lane);
        have = have + cnt < 32 * L ? have + cnt : 32 * L;
    }

    // Merge another sorted K-list stored at o[0..K) into this one.
    __device__ __forceinline__ void merge_list(const T* o, int lane) {
#pragma unroll
        for (int j = 0; j < L; ++j) lst[j] = kmax(lst[j], o[32 * L - 1 - (j * 32 + lane)]);
        bitonic_merge(lane);
    }
};

// Every kernel works on int32 words whose signed order is the key kind's
// order (KeyKind, topk_internal.h); ordered<KIND> maps an input word there
// and back (it is its own inverse):
//   kKeyI32  int32 values: unchanged;
//   kKeyU32  uint32 values: the top bit flipped (unsigned order -> signed);
//   kKeyF32  float32 bit patterns: the low 31 bits flipped when the sign is
//            set, so that signed order is IEEE 754 totalOrder (-NaN < -inf
//            < ... < -0 < +0 < ... < +inf < +NaN) -- the order of the "GPU
//            radix sort" page's float bit transform (its extensions
//            section), which maps that same order to unsigned integers.
template <int KIND>
__device__ __forceinline__ int ordered(int x) {
    if constexpr (KIND == kKeyU32) return x ^ INT_MIN;
    else if constexpr (KIND == kKeyF32) return x ^ ((x >> 31) & 0x7FFFFFFF);
    else return x;
}

template <int KIND>
__device__ __forceinline__ int4 ordered4(int4 v) {
    return make_int4(ordered<KIND>(v.x), ordered<KIND>(v.y), ordered<KIND>(v.z), ordered<KIND>(v.w));
}

__host__ __device__ __forceinline__ int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

}  // namespace topk

// ---------------------------------------------------------------------------
// Bulk asynchronous copies (TMA, non-tensor form) and mbarriers, for the
// streaming producer/consumer rings.  Every wait is bounded: it gives up after
// kWaitSpins tries and reports failure, so a kernel can never hang.
namespace topk {

constexpr int kWaitSpins = 1 << 22;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase of `bar` with the given parity has completed.
// Returns false if it did not within kWaitSpins tries.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (int i = 0; i < kWaitSpins; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// An L2 cache policy that marks lines as first to evict: for inputs read
// once, so that streaming them does not push out what the kernels that
// follow need (their code and small working arrays).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// A read-only 16-byte load with the L2 policy `policy` (see above).
__device__ __forceinline__ int4 ld_nc_hint(const int4* p, uint64_t policy) {
    int4 v;
    asm("ld.global.nc.L2::cache_hint.v4.s32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(policy));
    return v;
}

// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to this block's shared memory with the L2 policy `policy` (see above);
// completion is signalled on `bar`.
__device__ __forceinline__ void bulk_copy_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                   uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to this block's shared memory; completion is signalled on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic
// stream serialization (launch_pdl) may start while the previous kernel on
// the stream finishes; it must not touch anything that kernel writes until
// grid_dependency_wait() returns (which waits for the previous grid to
// complete and its writes to be visible), and it lets the next launch start
// with launch_dependents().  Both are hardware mechanisms, not spins.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` with programmatic stream serialization (see above).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace topk

namespace topk {
// Order this thread's earlier generic-proxy accesses to shared memory before
// its later async-proxy (bulk copy) accesses, e.g. before re-filling a stage
// whose contents the warp has just read.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
}  // namespace topk
