// int32 TopK: the k largest values of a large array, sorted descending.
//
// Method ("CUDA parallel optimisation: TopK, shared memory and two-stage
// reduction"): section 2.1 -- every block reduces its share of the input to
// k candidates (grid-stride loop, per-thread local top-k, shared-memory tree
// merge); section 2.2 -- a second single-block pass over the grid*k
// candidates gives the final k, identical to the CPU's answer.
//
// What is kept and what differs on sm_103a:
//   * Stage 1 streams 128-bit coalesced loads (8 in flight per lane) in a
//     persistent grid of 2 blocks/SM.  Instead of an insertion sort per
//     element, each warp compares every element once against a running k-th
//     value threshold; the rare survivors are compacted (ballot + popc) into
//     a per-warp shared-memory buffer, which is bitonic-sorted and cut back
//     to k when it fills, raising the threshold.
//   * Thresholds are shared: through shared memory inside the block and one
//     global word (atomicMax) across blocks.  Any threshold t used to
//     discard an element is one with at least k input elements >= t, and
//     every such t is published to the global word before the block
//     finishes.  Start values come from a sample: the k-th largest of group
//     maxima of the warp's first tile and of the array's last elements (the
//     latter keeps sorted-ascending input cheap).
//   * The block merge (section 2.1's tree) is a pairwise bitonic merge of
//     the warps' sorted lists.
//   * The second pass (section 2.2) runs in the same launch: the last block
//     to finish (atomic ticket, no waiting) selects the answer from the
//     grid*k candidates.  With t_g the final global threshold, the answer is
//     the candidates greater than t_g, sorted, padded with copies of t_g
//     when there are fewer than k of them.  If more candidates exceed t_g
//     than fit in shared memory, an 8-bit-digit radix select (the per-digit
//     histogram of "GPU radix sort", histogram section) finds the exact
//     k-th value first.
//   * The last block resets the two control words, so the next call on the
//     same workspace starts clean.  No block ever waits on another.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "topk_device.cuh"
#include "topk_internal.h"

namespace topk {

namespace {

constexpr int kU = 8;                 // 16-byte loads in flight per lane
constexpr int kTileVec = 32 * kU;     // int4 vectors per warp-tile (4 KiB)
constexpr int kTailVec = 64;          // int4 vectors in the tail sample (256 elements)

__device__ __forceinline__ unsigned bias(int v) { return (unsigned)v ^ 0x80000000u; }
__device__ __forceinline__ int unbias(unsigned u) { return (int)(u ^ 0x80000000u); }

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int ld_cg(const int* p) { return __ldcg(p); }

__device__ __forceinline__ int max4(int4 v) { return kmax(kmax(v.x, v.y), kmax(v.z, v.w)); }

// One warp-tile: kU int4 per lane, lane-interleaved so that every load
// instruction covers 512 contiguous bytes.  Vectors past nvec read as INT_MIN,
// which is never admitted (the filter is strict and thresholds are >= INT_MIN).
__device__ __forceinline__ void load_tile(int4 (&r)[kU], const int4* __restrict__ body, size_t nvec,
                                          size_t tile, int lane) {
    const size_t base = tile * kTileVec + lane;
    if (base + (kU - 1) * 32 < nvec) {
#pragma unroll
        for (int u = 0; u < kU; ++u) r[u] = __ldg(body + base + u * 32);
    } else {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const size_t i = base + u * 32;
            r[u] = i < nvec ? __ldg(body + i) : make_int4(INT_MIN, INT_MIN, INT_MIN, INT_MIN);
        }
    }
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

// Per-warp candidate buffer of capacity B in shared memory.
template <int B>
struct WarpBuf {
    int* buf;
    int cnt;   // warp-uniform number of entries
    int t;     // warp-uniform threshold: only values > t are admitted

    // Append the lanes' values that exceed t (order of arrival, compacted).
    __device__ __forceinline__ void admit(int v, int lane) {
        const bool p = v > t;
        const unsigned m = __ballot_sync(kFullMask, p);
        if (p) buf[cnt + __popc(m & lanemask_lt())] = v;
        cnt += __popc(m);
    }

    // Sort the buffer, keep its k largest, raise t to the k-th when there are
    // k of them.  Returns true when t was raised.
    __device__ bool flush(int k, int lane) {
        __syncwarp();
        bool raised = false;
        if constexpr (B == 256) {
            int v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int p = j * 32 + lane;
                v[j] = p < cnt ? buf[p] : INT_MIN;
            }
            warp_sort_desc<8>(v, lane);
            const int keep = cnt < k ? cnt : k;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int p = j * 32 + lane;
                if (p < keep) buf[p] = v[j];
            }
            if (cnt >= k) {
                const int kth = warp_sorted_at<8>(v, k - 1);
                if (kth > t) {
                    t = kth;
                    raised = true;
                }
            }
            cnt = keep;
        } else {
            for (int p = cnt + lane; p < B; p += 32) buf[p] = INT_MIN;
            __syncwarp();
            warp_sort_smem_desc(buf, B, lane);
            if (cnt >= k) {
                const int kth = buf[k - 1];
                if (kth > t) {
                    t = kth;
                    raised = true;
                }
            }
            cnt = cnt < k ? cnt : k;
        }
        __syncwarp();
        return raised;
    }
};

template <int B, int GL, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, (WARPS <= 8 ? 4 : 2) * (B <= 256 ? 1 : 0) + (B > 256 ? 1 : 0))
topk_i32_kernel(const int32_t* __restrict__ in, size_t n, int k, int32_t* __restrict__ out,
                int32_t* __restrict__ cand, I32Ctrl* __restrict__ ctrl) {
    extern __shared__ __align__(16) int smem[];
    __shared__ int s_thresh;
    __shared__ int s_last;
    __shared__ int s_count;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_thresh = INT_MIN;
    __syncthreads();

    // Split the array into an unaligned head (< 4 elements), a 16-byte
    // aligned body of int4 vectors and a scalar tail (< 4 elements).
    const uintptr_t addr = reinterpret_cast<uintptr_t>(in);
    size_t head = ((16u - (unsigned)(addr & 15u)) & 15u) >> 2;
    if (head > n) head = n;
    const int4* body = reinterpret_cast<const int4*>(in + head);
    const size_t nvec = (n - head) >> 2;
    const size_t tail0 = head + nvec * 4;
    const size_t ntiles = (nvec + kTileVec - 1) / kTileVec;
    const size_t gw = (size_t)blockIdx.x * WARPS + warp;
    const size_t nw = (size_t)gridDim.x * WARPS;

    WarpBuf<B> wb{smem + warp * B, 0, INT_MIN};
    int published = INT_MIN;  // the largest value this warp has sent to the global word

    auto publish = [&](int v) {
        if (lane == 0) {
            atomicMax(&s_thresh, v);
            if (v > published) atomicMax(&ctrl->thresh, bias(v));
        }
        published = kmax(published, v);
    };

    // Scalars outside the aligned body: at most 3 + 3 elements, taken by the
    // first warp of the grid.
    if (gw == 0) {
        const size_t ns = head + (n - tail0);
        const size_t pos = (size_t)lane < head ? (size_t)lane : tail0 + (lane - head);
        const int v = (size_t)lane < ns ? in[pos] : INT_MIN;
        wb.admit(v, lane);
    }

    bool first = true;
    for (size_t tile = gw; tile < ntiles; tile += nw) {
        const unsigned g = ld_relaxed_gpu(&ctrl->thresh);
        int4 r[kU];
        load_tile(r, body, nvec, tile, lane);

        if constexpr (GL > 0) {
          if (first) {
            first = false;
            // Start threshold: k-th largest group maximum of this tile and of
            // the array's last kTailVec vectors.
            int4 s[2];
            const long long tv = (long long)nvec - kTailVec + 2 * lane;
#pragma unroll
            for (int q = 0; q < 2; ++q)
                s[q] = tv + q >= 0 ? __ldg(body + tv + q) : make_int4(INT_MIN, INT_MIN, INT_MIN, INT_MIN);
            int seed = seed_from_groups<GL>(r, k, lane);
            if constexpr (GL <= 2) seed = kmax(seed, seed_from_groups<GL>(s, k, lane));
            if (seed > wb.t) {
                wb.t = seed;
                publish(seed);
            }
          }
        }

        wb.t = kmax(wb.t, kmax(unbias(g), *(volatile int*)&s_thresh));

        int m = INT_MIN;
#pragma unroll
        for (int u = 0; u < kU; ++u) m = kmax(m, max4(r[u]));
        if (__any_sync(kFullMask, m > wb.t)) {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (wb.cnt > B - 128) {
                    if (wb.flush(k, lane)) publish(wb.t);
                }
                wb.admit(r[u].x, lane);
                wb.admit(r[u].y, lane);
                wb.admit(r[u].z, lane);
                wb.admit(r[u].w, lane);
            }
        }
    }

    // Final per-warp list: sorted, k largest, padded with INT_MIN to K.
    if (wb.flush(k, lane)) publish(wb.t);
    const int K = next_pow2(k < 32 ? 32 : k);
    for (int p = wb.cnt + lane; p < K; p += 32) wb.buf[p] = INT_MIN;

    // Block merge: pairwise bitonic merges of sorted K-lists (section 2.1's
    // tree, with warps in place of threads).
#pragma unroll 1
    for (int s = 1; s < WARPS; s <<= 1) {
        __syncthreads();
        if ((warp & (2 * s - 1)) == 0) {
            int* a = smem + warp * B;
            const int* b = smem + (warp + s) * B;
            for (int i = lane; i < K; i += 32) a[i] = kmax(a[i], b[K - 1 - i]);
            __syncwarp();
            warp_merge_smem_desc(a, K, lane);
        }
    }
    __syncthreads();

    // Candidates of this block, and its k-th value as a threshold.
    for (int i = threadIdx.x; i < k; i += blockDim.x) cand[(size_t)blockIdx.x * k + i] = smem[i];
    if (threadIdx.x == 0) {
        const int kth = smem[k - 1];
        if (kth != INT_MIN) atomicMax(&ctrl->thresh, bias(kth));
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned ticket = atomicAdd(&ctrl->ticket, 1u);
        s_last = ticket == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;

    // ---- second stage, in the last block to finish ----------------------
    __threadfence();
    const int tg = unbias(ld_relaxed_gpu(&ctrl->thresh));
    const int cap = WARPS * B;
    int* list = smem;
    const size_t M = (size_t)gridDim.x * k;
    const size_t Mr = (M + blockDim.x - 1) / blockDim.x * blockDim.x;
    if (threadIdx.x == 0) s_count = 0;
    __syncthreads();
    for (size_t i = threadIdx.x; i < Mr; i += blockDim.x) {
        const int v = i < M ? ld_cg(cand + i) : INT_MIN;
        const bool p = v > tg;
        const unsigned m = __ballot_sync(kFullMask, p);
        int base = 0;
        if (lane == 0 && m) base = atomicAdd(&s_count, __popc(m));
        base = __shfl_sync(kFullMask, base, 0);
        const int pos = base + __popc(m & lanemask_lt());
        if (p && pos < cap) list[pos] = v;
    }
    __syncthreads();
    const int above = s_count;

    int T = tg;       // value that fills the places after the sorted list
    int nlist = above; // sorted entries that come first
    if (above > cap) {
        // Radix select over the candidates above tg: the exact k-th largest
        // value T, most significant 8-bit digit first.
        __shared__ unsigned hist[256];
        __shared__ unsigned s_prefix, s_need;
        unsigned prefix = 0, pmask = 0, need = (unsigned)k;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
            __syncthreads();
            for (size_t i = threadIdx.x; i < M; i += blockDim.x) {
                const int v = ld_cg(cand + i);
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
        if (threadIdx.x == 0) s_count = 0;
        __syncthreads();
        for (size_t i = threadIdx.x; i < Mr; i += blockDim.x) {
            const int v = i < M ? ld_cg(cand + i) : INT_MIN;
            const bool p = v > T;
            const unsigned m = __ballot_sync(kFullMask, p);
            int base = 0;
            if (lane == 0 && m) base = atomicAdd(&s_count, __popc(m));
            base = __shfl_sync(kFullMask, base, 0);
            if (p) list[base + __popc(m & lanemask_lt())] = v;
        }
        __syncthreads();
        nlist = s_count;
    }

    const int L = next_pow2(nlist < 2 ? 2 : nlist);
    for (int i = nlist + threadIdx.x; i < L; i += blockDim.x) list[i] = INT_MIN;
    block_sort_smem_desc(list, L);
    for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < nlist ? list[i] : T;
    if (threadIdx.x == 0) {
        ctrl->thresh = 0u;
        ctrl->ticket = 0u;
    }
}

template <int B, int GL, int WARPS>
struct I32Variant {
    static constexpr int kWarps = WARPS;
    static size_t smem_bytes() { return (size_t)WARPS * B * sizeof(int); }
    static const void* fn() { return reinterpret_cast<const void*>(&topk_i32_kernel<B, GL, WARPS>); }
    static void launch(int grid, cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out,
                       int32_t* cand, I32Ctrl* ctrl) {
        topk_i32_kernel<B, GL, WARPS><<<grid, WARPS * 32, smem_bytes(), s>>>(in, n, k, out, cand, ctrl);
    }
};

using VarK32 = I32Variant<256, 1, 16>;
using VarK64 = I32Variant<256, 2, 16>;
using VarK128 = I32Variant<256, 4, 16>;
using VarK1024 = I32Variant<2048, 0, 16>;

template <class V>
cudaError_t plan_for(int device, size_t n, I32Plan* plan) {
    int sms = 0, per_sm = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    const size_t smem = V::smem_bytes();
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(V::fn(), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, V::fn(), V::kWarps * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const size_t nvec = n / 4;
    const size_t tiles = (nvec + kTileVec - 1) / kTileVec;
    const size_t want = (tiles + V::kWarps - 1) / V::kWarps;
    size_t grid = (size_t)sms * per_sm;
    if (want < grid) grid = want;
    if (grid < 1) grid = 1;
    plan->grid = (int)grid;
    plan->max_grid = sms * per_sm;
    return cudaSuccess;
}

}  // namespace

cudaError_t i32_plan(int device, size_t n, int k, I32Plan* plan) {
    if (k <= 32) return plan_for<VarK32>(device, n, plan);
    if (k <= 64) return plan_for<VarK64>(device, n, plan);
    if (k <= 128) return plan_for<VarK128>(device, n, plan);
    return plan_for<VarK1024>(device, n, plan);
}

cudaError_t i32_launch(const I32Plan& plan, cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out,
                       int32_t* cand, I32Ctrl* ctrl) {
    if (k <= 32)
        VarK32::launch(plan.grid, s, in, n, k, out, cand, ctrl);
    else if (k <= 64)
        VarK64::launch(plan.grid, s, in, n, k, out, cand, ctrl);
    else if (k <= 128)
        VarK128::launch(plan.grid, s, in, n, k, out, cand, ctrl);
    else
        VarK1024::launch(plan.grid, s, in, n, k, out, cand, ctrl);
    return cudaGetLastError();
}

}  // namespace topk
