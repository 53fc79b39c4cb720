// int32 TopK for large k: radix select.
//
// The filter of the streaming kernels keeps one list of k candidates per
// warp, which stops paying for itself once k is in the hundreds.  For
// 128 < k <= 32768 the selection is a radix select on the order-preserving
// key u = value ^ 0x80000000 ("GPU radix sort": per-block shared-memory
// digit histograms, its histogram section; the digit width is widened from
// 8 to 12 bits because a select needs only the bucket that holds the k-th
// value, not a full reordering):
//   pass 1   histogram of the top 12 bits of every key; the last block to
//            finish finds the bucket b1 holding the k-th largest key.
//   pass 2   keys whose top 12 bits exceed b1 are in the answer: they are
//            collected.  Keys in bucket b1 are histogrammed on the next 12
//            bits and copied to a boundary buffer while it has room.  The
//            last block finds the bucket b2 of the k-th key there.
//   pass 3   only if the buffer overflowed: keys in b1 above b2 are
//            collected; keys in (b1, b2) are histogrammed on the last 8
//            bits, which fixes the k-th key T exactly.
//   final    one block: if the buffer holds all of bucket b1, it finds the
//            k-th key inside it (two more histogram levels); the answer is
//            every collected key plus the buffered keys above T, sorted,
//            padded with copies of T.
// Each pass's decisions stay on the device (the last block writes them to
// the control words), so the call stays asynchronous: pass 3 starts, reads
// that it is not needed, and returns.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "topk_device.cuh"
#include "topk_internal.h"

namespace topk {

namespace {

constexpr int kRThreads = 512;
constexpr int kRU = 8;        // 16-byte loads in flight per thread
constexpr int kBins = 4096;   // 12-bit digits
constexpr int kFinalThreads = 1024;

struct RadixCtrl {
    unsigned ticket;     // blocks finished in the current pass
    unsigned prefix;     // fixed high bits of the k-th key so far
    unsigned level;      // digits fixed so far: 1 (12 bits), 2 (24), 3 (32)
    unsigned need;       // keys with the current prefix that belong to the answer
    unsigned ncand;      // keys collected (certainly in the answer)
    unsigned nbnd;       // keys appended to the boundary buffer (may exceed its capacity)
    unsigned bucket;     // size of the current boundary bucket
    unsigned pad[57];
};
static_assert(sizeof(RadixCtrl) == 256, "one line");

struct RadixView {
    unsigned* status;
    RadixCtrl* ctrl;
    unsigned* hist;  // kBins global counts
    unsigned* cand;  // collected keys (fewer than k)
    unsigned* bnd;   // boundary buffer
};

__device__ __forceinline__ RadixView radix_view(unsigned char* base, int k) {
    RadixView v;
    v.status = reinterpret_cast<unsigned*>(base + kI32StatusOffset);
    v.ctrl = reinterpret_cast<RadixCtrl*>(base + kRadixCtrlOffset);
    v.hist = reinterpret_cast<unsigned*>(base + kRadixHistOffset);
    v.cand = reinterpret_cast<unsigned*>(base + kRadixCandOffset);
    v.bnd = v.cand + ((size_t)k + 63) / 64 * 64;
    return v;
}

__device__ __forceinline__ unsigned key_of(int v) { return (unsigned)v ^ 0x80000000u; }

// Add one to bin d of a shared histogram for every lane with `has`; a warp
// whose lanes all hit one bin (sorted or duplicate-heavy input) adds once.
__device__ __forceinline__ void hist_add(unsigned* h, unsigned d, bool has) {
    const unsigned m = __ballot_sync(kFullMask, has);
    if (!m) return;
    const int leader = __ffs(m) - 1;
    const unsigned d0 = __shfl_sync(kFullMask, d, leader);
    if (__all_sync(kFullMask, !has || d == d0)) {
        if ((threadIdx.x & 31) == leader) atomicAdd(&h[d0], (unsigned)__popc(m));
    } else if (has) {
        atomicAdd(&h[d], 1u);
    }
}

// Append the lanes' keys with `p` to dst[*counter ...] (warp-aggregated);
// slots at or past cap are counted but not written.
__device__ __forceinline__ void append(unsigned* dst, unsigned* counter, size_t cap, unsigned u, bool p) {
    const unsigned m = __ballot_sync(kFullMask, p);
    if (!m) return;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(m) - 1;
    unsigned base = 0;
    if (lane == leader) base = atomicAdd(counter, (unsigned)__popc(m));
    base = __shfl_sync(kFullMask, base, leader);
    if (p) {
        const unsigned slot = base + __popc(m & lanemask_lt());
        if (slot < cap) dst[slot] = u;
    }
}

// Block-level: merge the shared histogram into the global one, take a
// ticket; true in the last block to finish.
__device__ bool hist_done(const RadixView& rv, const unsigned* sh, int* s_last) {
    __syncthreads();
    for (int i = threadIdx.x; i < kBins; i += blockDim.x)
        if (sh[i]) atomicAdd(&rv.hist[i], sh[i]);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *s_last = atomicAdd(&rv.ctrl->ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (*s_last) __threadfence();
    return *s_last != 0;
}

// Last block of a pass: find the bucket of the need-th largest key in the
// global histogram (nbins bins, highest first), fix its digit into the
// prefix, clear the histogram and the ticket.
__device__ void pick_bucket(const RadixView& rv, int nbins, int shift, unsigned need, unsigned prefix,
                            unsigned* s_scan, bool keep_hist) {
    // Suffix sums from the top, one warp per 32-bin chunk is plenty here:
    // thread 0 walks the bins (at most 4096).
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned acc = 0;
        int d = nbins - 1;
        for (; d > 0; --d) {
            const unsigned c = __ldcg(&rv.hist[d]);
            if (acc + c >= need) break;
            acc += c;
        }
        s_scan[0] = (unsigned)d;
        s_scan[1] = acc;                      // keys above the bucket
        s_scan[2] = __ldcg(&rv.hist[d]);      // keys in the bucket
    }
    __syncthreads();
    if (!keep_hist)
        for (int i = threadIdx.x; i < nbins; i += blockDim.x) rv.hist[i] = 0u;
    if (threadIdx.x == 0) {
        rv.ctrl->prefix = prefix | (s_scan[0] << shift);
        rv.ctrl->need = need - s_scan[1];
        rv.ctrl->bucket = s_scan[2];
        rv.ctrl->level += 1;
        rv.ctrl->ticket = 0u;
    }
}

// Streaming helper: every thread visits its int4 vectors of the aligned
// body in batches of kRU (coalesced), plus the < 8 scalars outside it, and
// calls f(key, valid) for each of its elements with warp-uniform control.
template <class F>
__device__ __forceinline__ void for_each_key(const int32_t* __restrict__ in, size_t n, F f) {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(in);
    size_t head = ((16u - (unsigned)(addr & 15u)) & 15u) >> 2;
    if (head > n) head = n;
    const int4* body = reinterpret_cast<const int4*>(in + head);
    const size_t nvec = (n - head) >> 2;
    const size_t tail0 = head + nvec * 4;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t base = (size_t)blockIdx.x * blockDim.x * kRU; base < nvec; base += stride * kRU) {
        int4 r[kRU];
#pragma unroll
        for (int u = 0; u < kRU; ++u) {
            const size_t i = base + (size_t)u * blockDim.x + threadIdx.x;
            r[u] = i < nvec ? __ldg(body + i) : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kRU; ++u) {
            const bool ok = base + (size_t)u * blockDim.x + threadIdx.x < nvec;
            f(key_of(r[u].x), ok);
            f(key_of(r[u].y), ok);
            f(key_of(r[u].z), ok);
            f(key_of(r[u].w), ok);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < 32) {
        const size_t ns = head + (n - tail0);
        const size_t lane = threadIdx.x;
        const size_t pos = lane < head ? lane : tail0 + (lane - head);
        f(lane < ns ? key_of(in[pos]) : 0u, lane < ns);
    }
}

__global__ void __launch_bounds__(kRThreads, 2)
radix_pass1_kernel(const int32_t* __restrict__ in, size_t n, int k, unsigned char* __restrict__ scratch) {
    __shared__ unsigned sh[kBins];
    __shared__ int s_last;
    __shared__ unsigned s_scan[4];
    const RadixView rv = radix_view(scratch, k);
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
    for_each_key(in, n, [&](unsigned u, bool ok) { hist_add(sh, u >> 20, ok); });
    if (hist_done(rv, sh, &s_last)) {
        if (threadIdx.x == 0) {
            rv.ctrl->level = 0u;
            rv.ctrl->ncand = 0u;
            rv.ctrl->nbnd = 0u;
        }
        pick_bucket(rv, kBins, 20, (unsigned)k, 0u, s_scan, false);
    }
}

// Pass 2 (level 2) and pass 3 (level 3); see the file comment.
__global__ void __launch_bounds__(kRThreads, 2)
radix_collect_kernel(const int32_t* __restrict__ in, size_t n, int k, unsigned char* __restrict__ scratch,
                     size_t cap, int level) {
    __shared__ unsigned sh[kBins];
    __shared__ int s_last;
    __shared__ unsigned s_scan[4];
    __shared__ unsigned s_prefix, s_go;
    const RadixView rv = radix_view(scratch, k);
    if (threadIdx.x == 0) {
        const unsigned lv = __ldcg(&rv.ctrl->level);
        s_prefix = __ldcg(&rv.ctrl->prefix);
        // Pass 3 runs only if pass 2's buffer could not hold bucket b1.
        s_go = level == 2 ? (lv == 1) : (lv == 2 && __ldcg(&rv.ctrl->nbnd) > cap);
    }
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
    if (!s_go) return;
    const unsigned prefix = s_prefix;
    if (level == 2) {
        // prefix: top 12 bits fixed.
        for_each_key(in, n, [&](unsigned u, bool ok) {
            const unsigned hi = u & 0xFFF00000u;
            append(rv.cand, &rv.ctrl->ncand, (size_t)k, u, ok && hi > prefix);
            const bool b = ok && hi == prefix;
            hist_add(sh, (u >> 8) & 0xFFFu, b);
            append(rv.bnd, &rv.ctrl->nbnd, cap, u, b);
        });
    } else {
        // prefix: top 24 bits fixed (bucket b1, then b2).
        for_each_key(in, n, [&](unsigned u, bool ok) {
            const bool in_b1 = ok && (u & 0xFFF00000u) == (prefix & 0xFFF00000u);
            append(rv.cand, &rv.ctrl->ncand, (size_t)k, u, in_b1 && (u & 0xFFFFFF00u) > prefix);
            hist_add(sh, u & 0xFFu, in_b1 && (u & 0xFFFFFF00u) == prefix);
        });
    }
    if (hist_done(rv, sh, &s_last)) {
        const unsigned need = __ldcg(&rv.ctrl->need);
        if (level == 2)
            pick_bucket(rv, kBins, 8, need, prefix, s_scan, false);
        else
            pick_bucket(rv, 256, 0, need, prefix, s_scan, true);  // the final step reads it
    }
}

// Final: one block.  Shared memory: the sort area (next_pow2(k) ints) and a
// histogram.
__global__ void __launch_bounds__(kFinalThreads, 1)
radix_final_kernel(int k, int32_t* __restrict__ out, unsigned char* __restrict__ scratch, size_t cap) {
    extern __shared__ __align__(16) unsigned s_list[];
    __shared__ unsigned sh[kBins];
    __shared__ unsigned s_scan[4];
    __shared__ unsigned s_n;
    const RadixView rv = radix_view(scratch, k);
    const unsigned level = __ldcg(&rv.ctrl->level);
    const unsigned ncand = __ldcg(&rv.ctrl->ncand);
    const unsigned nbnd = __ldcg(&rv.ctrl->nbnd);
    unsigned prefix = __ldcg(&rv.ctrl->prefix);
    unsigned need = __ldcg(&rv.ctrl->need);

    unsigned T;             // the k-th largest key
    bool from_buffer;       // keys above T still to be taken from the buffer
    if (level == 3) {
        T = prefix;         // all 32 bits fixed; the collected keys are exactly those above T
        from_buffer = false;
    } else {
        // level 2: the buffer holds every key of bucket b1 (top 12 bits);
        // the k-th key is the need-th largest of the buffer's keys whose
        // next 12 bits equal b2.  Resolve the last 8 bits with one more
        // histogram over the buffer.
        const unsigned nb = nbnd < cap ? nbnd : (unsigned)cap;
        for (int i = threadIdx.x; i < 256; i += blockDim.x) sh[i] = 0u;
        __syncthreads();
        for (unsigned i = threadIdx.x; i < nb; i += blockDim.x) {
            const unsigned u = __ldcg(&rv.bnd[i]);
            if ((u & 0xFFFFFF00u) == prefix) atomicAdd(&sh[u & 0xFFu], 1u);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned acc = 0;
            int d = 255;
            for (; d > 0; --d) {
                if (acc + sh[d] >= need) break;
                acc += sh[d];
            }
            s_scan[0] = prefix | (unsigned)d;
        }
        __syncthreads();
        T = s_scan[0];
        from_buffer = true;
    }

    // Everything above T: the collected keys, then (level 2) the buffered
    // keys above T, or (level 3) the keys of the last 24-bit bucket whose
    // low byte exceeds T's -- their values and counts are exactly the
    // histogram bins above T's byte.  Fewer than k in all.
    if (threadIdx.x == 0) s_n = 0;
    __syncthreads();
    const unsigned nc = ncand < (unsigned)k ? ncand : (unsigned)k;
    for (unsigned i = threadIdx.x; i < nc; i += blockDim.x) s_list[i] = __ldcg(&rv.cand[i]);
    if (threadIdx.x == 0) s_n = nc;
    __syncthreads();
    if (!from_buffer) {
        if (threadIdx.x == 0) {
            unsigned at = s_n;
            for (unsigned d = (T & 0xFFu) + 1; d < 256; ++d) {
                const unsigned c = __ldcg(&rv.hist[d]);
                for (unsigned j = 0; j < c && at < (unsigned)k; ++j) s_list[at++] = (T & 0xFFFFFF00u) | d;
            }
            s_n = at;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < 256; i += blockDim.x) rv.hist[i] = 0u;
    }
    if (from_buffer) {
        const unsigned nb = nbnd < cap ? nbnd : (unsigned)cap;
        const unsigned nbr = (nb + blockDim.x - 1) / blockDim.x * blockDim.x;
        for (unsigned i = threadIdx.x; i < nbr; i += blockDim.x) {
            const unsigned u = i < nb ? __ldcg(&rv.bnd[i]) : 0u;
            const bool p = i < nb && u > T;
            const unsigned m = __ballot_sync(kFullMask, p);
            unsigned base = 0;
            const int lane = threadIdx.x & 31;
            if (lane == 0 && m) base = atomicAdd(&s_n, (unsigned)__popc(m));
            base = __shfl_sync(kFullMask, base, 0);
            if (p) {
                const unsigned slot = base + __popc(m & lanemask_lt());
                if (slot < (unsigned)k) s_list[slot] = u;
            }
        }
        __syncthreads();
    }
    unsigned nlist = s_n < (unsigned)k ? s_n : (unsigned)k;
    const int L = next_pow2((int)(nlist < 2 ? 2 : nlist));
    for (int i = (int)nlist + threadIdx.x; i < L; i += blockDim.x) s_list[i] = 0u;
    block_sort_smem_desc(s_list, L);
    for (int i = threadIdx.x; i < k; i += blockDim.x)
        out[i] = (int32_t)(((unsigned)i < nlist ? s_list[i] : T) ^ 0x80000000u);
    // Leave the control words zero, as every int32 plan expects them.
    if (threadIdx.x < 7) reinterpret_cast<unsigned*>(rv.ctrl)[threadIdx.x] = 0u;
}

struct RadixFit {
    int grid = 0;
};

cudaError_t radix_fit(int device, RadixFit* out) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static RadixFit cache[kMaxDev];
    if (device < 0 || device >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[device].grid == 0) {
        int sms = 0, a = 0, b = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, reinterpret_cast<const void*>(&radix_pass1_kernel),
                                                          kRThreads, 0);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, reinterpret_cast<const void*>(&radix_collect_kernel),
                                                          kRThreads, 0);
        if (e != cudaSuccess) return e;
        const int per_sm = a < b ? a : b;
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&radix_final_kernel),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kRadixMaxK * sizeof(unsigned)));
        if (e != cudaSuccess) return e;
        cache[device].grid = sms * (per_sm < 1 ? 1 : per_sm);
    }
    *out = cache[device];
    return cudaSuccess;
}

}  // namespace

cudaError_t radix_launch(cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out, void* scratch,
                         size_t cap) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    RadixFit f;
    e = radix_fit(device, &f);
    if (e != cudaSuccess) return e;
    const size_t per_block = (size_t)kRThreads * kRU * 4;
    size_t grid = (n + per_block - 1) / per_block;
    if (grid > (size_t)f.grid) grid = f.grid;
    if (grid < 1) grid = 1;
    auto* sc = static_cast<unsigned char*>(scratch);
    radix_pass1_kernel<<<(int)grid, kRThreads, 0, s>>>(in, n, k, sc);
    radix_collect_kernel<<<(int)grid, kRThreads, 0, s>>>(in, n, k, sc, cap, 2);
    radix_collect_kernel<<<(int)grid, kRThreads, 0, s>>>(in, n, k, sc, cap, 3);
    const size_t smem = (size_t)next_pow2(k) * sizeof(unsigned);
    radix_final_kernel<<<1, kFinalThreads, smem, s>>>(k, out, sc, cap);
    return cudaGetLastError();
}

}  // namespace topk
