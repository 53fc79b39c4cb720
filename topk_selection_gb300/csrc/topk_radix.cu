// int32 TopK for large k: a sampled threshold, one filtering pass over the
// input, a cluster-wide radix select and a range-partitioned sort.
//
// The filter of the streaming kernels keeps one register list of k
// candidates per warp, which stops paying once k is in the hundreds.  For
// 128 < k <= 32768 the selection runs on the order-preserving key
// u = value ^ 0x80000000 (unsigned order = signed order) and uses the digit
// histograms of "GPU radix sort" (per-block shared-memory histograms, its
// histogram section), with 12-bit digits: a select needs only the bucket
// that holds the k-th key, not a reordering.
//
// Plan when n exceeds what one cluster holds (kRadixClusterCap keys):
//   sample   one cluster of 8 CTAs gathers 2^18 keys from 16384 evenly
//            spaced 16-element segments and selects the j-th largest, j a few
//            standard deviations above k's expected share of the sample.
//            That key is the filter threshold t.
//   filter   a persistent grid reads the input once: keys above t go to the
//            candidate buffer, keys equal to t are counted.  The last block
//            to finish decides what follows:
//              buffer count >= k and it fits   -> select the k-th in the buffer
//              buffer + equal count >= k       -> t is the k-th key
//              otherwise                       -> the exact passes
//   exact    three grid passes that do work only when the sample misled the
//            filter; otherwise each reads the state word and returns:
//              pass 1   12-bit histogram of the top bits -> bucket b1
//              pass 2   if every key at or above b1 fits the buffer, collect
//                       them (then select in the buffer); else histogram the
//                       next 12 bits of the keys in b1 -> bucket b2
//              pass 3   collect the keys above the 24-bit prefix and
//                       histogram the low 8 bits of the keys in it; that
//                       fixes the k-th key T, and the keys between T and the
//                       prefix's top are written from the histogram
//   final    one cluster loads the buffer into its 8 CTAs' shared memory and
//            selects the k-th key with four cluster-wide 8-bit digit
//            histograms (summed through distributed shared memory).  Each CTA
//            keeps its keys above the k-th; rank 0 cuts their value range into
//            about 768-key ranges from a sample weighted by each CTA's share
//            (a value that dominates the sample gets a range of its own).
//   sort     one CTA per range: it counts the keys in higher ranges for its
//            output offset, gathers its own and sorts them in shared memory.
//            The cluster writes the copies of the k-th key after them.
// When n fits one cluster, the cluster kernel and the sort alone run, on the
// input itself.
// Every decision stays on the device, so a call only enqueues work.  No
// kernel here waits on another block or CTA except through hardware
// barriers (__syncthreads, the cluster barrier), so none can hang.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "topk_device.cuh"
#include "topk_internal.h"

namespace topk {

namespace {

constexpr int kRThreads = 512;  // grid passes
constexpr int kRU = 8;          // 16-byte loads in flight per thread
constexpr int kBins = 4096;     // 12-bit digits

constexpr int kClCtas = 8;  // CTAs per cluster (portable size)
constexpr int kClThreads = 1024;
constexpr int kClWarps = kClThreads / 32;
constexpr int kClSlice = 32768;  // keys per CTA
constexpr unsigned kSegLen = 16;
constexpr unsigned kSegments = (unsigned)(kRadixClusterCap / kSegLen);
static_assert((size_t)kClCtas * kClSlice == kRadixClusterCap, "cluster capacity");
static_assert(kClSlice == kClWarps * 1024, "a warp owns a 1024-key sub-slice");

enum : unsigned { kStatePending = 0, kStateSelect = 1, kStateSorted = 2, kStateExact = 3 };
enum : unsigned { kExactCollectAll = 1, kExactHistogram = 2 };

// Control words of the radix plan; zero between launches (the final zeroes
// the first kCtrlWords words).
struct RadixCtrl {
    unsigned ticket;          // blocks finished in the current grid pass
    unsigned state;           // kState*: what the later kernels do
    unsigned t;               // filter threshold key; after pass 3, the k-th key
    unsigned prefix;          // exact passes: digits fixed so far
    unsigned need;            // exact passes: keys with that prefix still to take
    unsigned exact_mode;      // kExact*: what pass 2 does
    unsigned long long nbuf;  // keys appended to the buffer (counts past its capacity)
    unsigned long long neq;   // keys equal to t seen by the filter
    unsigned pad[54];
};
static_assert(sizeof(RadixCtrl) == 256, "one line");
constexpr int kCtrlWords = 10;

struct RadixView {
    RadixCtrl* ctrl;
    unsigned long long* hist;  // kBins global counts
    unsigned* buf;             // candidate buffer
};

__device__ __forceinline__ RadixView radix_view(unsigned char* base) {
    RadixView v;
    v.ctrl = reinterpret_cast<RadixCtrl*>(base + kRadixCtrlOffset);
    v.hist = reinterpret_cast<unsigned long long*>(base + kRadixHistOffset);
    v.buf = reinterpret_cast<unsigned*>(base + kRadixBufOffset);
    return v;
}

__device__ __forceinline__ unsigned key_of(int v) { return (unsigned)v ^ 0x80000000u; }
__device__ __forceinline__ int32_t value_of(unsigned u) { return (int32_t)(u ^ 0x80000000u); }

// Sum of v over the threads above this one in the block (thread order is
// bin order: higher threads hold higher bins).  s_warp: 64 slots.
template <typename T>
__device__ __forceinline__ T block_suffix_excl(T v, T* s_warp) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T y = __shfl_down_sync(kFullMask, x, o);
        if (lane + o < 32) x += y;
    }
    if (lane == 0) s_warp[w] = x;
    __syncthreads();
    if (w == 0) {
        const T own = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : T(0);
        T z = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const T y = __shfl_down_sync(kFullMask, z, o);
            if (lane + o < 32) z += y;
        }
        s_warp[32 + lane] = z - own;
    }
    __syncthreads();
    return (x - v) + s_warp[32 + w];
}

// ---------------------------------------------------------------------------
// Grid passes

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

// Keys appended to the candidate buffer through a per-warp shared stage,
// 32 at a time: one global atomic per 32 keys.  Slots at or past cap are
// counted but not written; once the buffer has overflowed the warp stops
// appending (the plan then takes the exact passes anyway).
struct WarpAppender {
    unsigned* st;  // this warp's 64 stage slots
    unsigned cnt;  // keys staged (warp-uniform)
    bool full;     // the buffer overflowed (warp-uniform)

    __device__ __forceinline__ void push(const RadixView& rv, unsigned cap, unsigned u, bool p) {
        const unsigned m = __ballot_sync(kFullMask, p);
        if (!m || full) return;
        const int lane = threadIdx.x & 31;
        if (p) st[cnt + __popc(m & lanemask_lt())] = u;
        cnt += __popc(m);
        if (cnt >= 32) {
            __syncwarp();
            unsigned long long base = 0;
            if (lane == 0) base = atomicAdd(&rv.ctrl->nbuf, 32ull);
            base = __shfl_sync(kFullMask, base, 0);
            if (base + lane < cap) rv.buf[base + lane] = st[lane];
            const unsigned rest = cnt - 32;
            const unsigned v = (unsigned)lane < rest ? st[32 + lane] : 0u;
            __syncwarp();
            if ((unsigned)lane < rest) st[lane] = v;
            __syncwarp();
            cnt = rest;
            full = base + 32 > cap;
        }
    }

    __device__ __forceinline__ void flush(const RadixView& rv, unsigned cap) {
        if (!cnt || full) return;
        const int lane = threadIdx.x & 31;
        __syncwarp();
        unsigned long long base = 0;
        if (lane == 0) base = atomicAdd(&rv.ctrl->nbuf, (unsigned long long)cnt);
        base = __shfl_sync(kFullMask, base, 0);
        if ((unsigned)lane < cnt && base + lane < cap) rv.buf[base + lane] = st[lane];
        cnt = 0;
    }
};

// Input walk shared by the grid passes: every thread visits its int4 vectors
// of the 16-byte-aligned body in batches of kRU (coalesced); f_vec(v, ok) is
// called per vector with warp-uniform control.  The < 8 scalars outside the
// body go to warp 0 of block 0 through f_tail(value, ok), one per lane.
template <class FV, class FT>
__device__ __forceinline__ void for_each_vec(const int32_t* __restrict__ in, size_t n, FV f_vec, FT f_tail) {
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
        for (int u = 0; u < kRU; ++u) f_vec(r[u], base + (size_t)u * blockDim.x + threadIdx.x < nvec);
    }
    if (blockIdx.x == 0 && threadIdx.x < 32) {
        const size_t ns = head + (n - tail0);
        const size_t lane = threadIdx.x;
        const size_t pos = lane < head ? lane : tail0 + (lane - head);
        f_tail(lane < ns ? in[pos] : 0, lane < ns);
    }
}

template <class F>
__device__ __forceinline__ void for_each_key(const int32_t* __restrict__ in, size_t n, F f) {
    for_each_vec(
        in, n,
        [&](const int4& v, bool ok) {
            f(key_of(v.x), ok);
            f(key_of(v.y), ok);
            f(key_of(v.z), ok);
            f(key_of(v.w), ok);
        },
        [&](int v, bool ok) { f(key_of(v), ok); });
}

// Block-level end of a grid pass: merge the shared histogram (if any) into
// the global one, take a ticket; true in the last block to finish.
__device__ bool pass_done(const RadixView& rv, const unsigned* sh, int* s_last) {
    __syncthreads();
    if (sh)
        for (int i = threadIdx.x; i < kBins; i += blockDim.x)
            if (sh[i]) atomicAdd(&rv.hist[i], (unsigned long long)sh[i]);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *s_last = atomicAdd(&rv.ctrl->ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (*s_last) __threadfence();
    return *s_last != 0;
}

struct Bucket {
    unsigned digit;            // bucket holding the need-th largest key
    unsigned above;            // keys in higher buckets (< need)
    unsigned long long count;  // keys in the bucket
};

// Last block of a grid pass: find the bucket of the need-th largest key in
// the global histogram (nbins bins, at most 8 per thread), then clear the
// histogram and the ticket.  s_scan: 64 slots; s_pick: the result, for
// every thread.
__device__ void pick_bucket(const RadixView& rv, int nbins, unsigned need, unsigned long long* s_scan,
                            Bucket* s_pick) {
    const int per = nbins >= (int)blockDim.x ? nbins / (int)blockDim.x : 1;
    const int first = threadIdx.x * per;
    unsigned long long c[8];
    unsigned long long tot = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        c[b] = (b < per && first + b < nbins) ? __ldcg(&rv.hist[first + b]) : 0ull;
        tot += c[b];
    }
    const unsigned long long above = block_suffix_excl(tot, s_scan);
    if (above < need && need <= above + tot) {
        unsigned long long acc = above;
#pragma unroll
        for (int b = 7; b >= 0; --b) {
            if (b < per && acc + c[b] >= need) {
                s_pick->digit = (unsigned)(first + b);
                s_pick->above = (unsigned)acc;
                s_pick->count = c[b];
                break;
            }
            acc += c[b];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nbins; i += blockDim.x) rv.hist[i] = 0ull;
    if (threadIdx.x == 0) rv.ctrl->ticket = 0u;
    __syncthreads();
}

// The filter: keys above t to the buffer, keys equal to t counted.
__global__ void __launch_bounds__(kRThreads, 2)
radix_filter_kernel(const int32_t* __restrict__ in, size_t n, int k, unsigned char* __restrict__ scratch,
                    unsigned cap) {
    __shared__ unsigned stage[kRThreads / 32][64];
    __shared__ unsigned long long s_neq;
    __shared__ int s_last;
    const RadixView rv = radix_view(scratch);
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) s_neq = 0ull;
    const int tv = value_of(__ldcg(&rv.ctrl->t));
    WarpAppender ap{stage[threadIdx.x >> 5], 0u, false};
    unsigned neq = 0;
    auto visit = [&](int v, bool ok) {
        neq += (ok && v == tv) ? 1u : 0u;
        ap.push(rv, cap, key_of(v), ok && v > tv);
    };
    for_each_vec(
        in, n,
        [&](const int4& v, bool ok) {
            const int mx = max(max(v.x, v.y), max(v.z, v.w));
            if (__any_sync(kFullMask, ok && mx >= tv) && !ap.full) {
                visit(v.x, ok);
                visit(v.y, ok);
                visit(v.z, ok);
                visit(v.w, ok);
            }
        },
        visit);
    ap.flush(rv, cap);
    neq = __reduce_add_sync(kFullMask, neq);
    __syncthreads();
    if (lane == 0 && neq) atomicAdd(&s_neq, (unsigned long long)neq);
    __syncthreads();
    if (threadIdx.x == 0 && s_neq) atomicAdd(&rv.ctrl->neq, s_neq);
    if (pass_done(rv, nullptr, &s_last) && threadIdx.x == 0) {
        const unsigned long long nb = atomicAdd(&rv.ctrl->nbuf, 0ull);
        const unsigned long long ne = atomicAdd(&rv.ctrl->neq, 0ull);
        unsigned st = kStateExact;
        if (nb <= cap && nb >= (unsigned long long)k)
            st = kStateSelect;
        else if (nb <= cap && nb + ne >= (unsigned long long)k)
            st = kStateSorted;
        rv.ctrl->state = st;
        rv.ctrl->ticket = 0u;
    }
}

// Exact pass 1: 12-bit histogram of the top bits; the last block picks b1
// and decides whether pass 2 can collect every key at or above it.
__global__ void __launch_bounds__(kRThreads, 2)
radix_exact1_kernel(const int32_t* __restrict__ in, size_t n, int k, unsigned char* __restrict__ scratch,
                    unsigned cap) {
    __shared__ unsigned sh[kBins];
    __shared__ unsigned long long s_scan[64];
    __shared__ Bucket s_pick;
    __shared__ int s_last, s_go;
    const RadixView rv = radix_view(scratch);
    if (threadIdx.x == 0) s_go = __ldcg(&rv.ctrl->state) == kStateExact;
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
    if (!s_go) return;
    for_each_key(in, n, [&](unsigned u, bool ok) { hist_add(sh, u >> 20, ok); });
    if (pass_done(rv, sh, &s_last)) {
        pick_bucket(rv, kBins, (unsigned)k, s_scan, &s_pick);
        if (threadIdx.x == 0) {
            rv.ctrl->prefix = s_pick.digit << 20;
            rv.ctrl->need = (unsigned)k - s_pick.above;
            rv.ctrl->exact_mode = s_pick.above + s_pick.count <= cap ? kExactCollectAll : kExactHistogram;
            rv.ctrl->nbuf = 0ull;
            rv.ctrl->neq = 0ull;
        }
    }
}

// Exact pass 2: collect every key at or above b1, or histogram the next 12
// bits of the keys in b1.
__global__ void __launch_bounds__(kRThreads, 2)
radix_exact2_kernel(const int32_t* __restrict__ in, size_t n, unsigned char* __restrict__ scratch, unsigned cap) {
    __shared__ unsigned sh[kBins];
    __shared__ unsigned stage[kRThreads / 32][64];
    __shared__ unsigned long long s_scan[64];
    __shared__ Bucket s_pick;
    __shared__ int s_last, s_go;
    __shared__ unsigned s_prefix, s_mode, s_need;
    const RadixView rv = radix_view(scratch);
    if (threadIdx.x == 0) {
        s_go = __ldcg(&rv.ctrl->state) == kStateExact;
        s_prefix = __ldcg(&rv.ctrl->prefix);
        s_mode = __ldcg(&rv.ctrl->exact_mode);
        s_need = __ldcg(&rv.ctrl->need);
    }
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
    if (!s_go) return;
    const unsigned prefix = s_prefix;
    const bool collect = s_mode == kExactCollectAll;
    if (collect) {
        WarpAppender ap{stage[threadIdx.x >> 5], 0u, false};
        for_each_key(in, n, [&](unsigned u, bool ok) { ap.push(rv, cap, u, ok && (u & 0xFFF00000u) >= prefix); });
        ap.flush(rv, cap);
    } else {
        for_each_key(in, n, [&](unsigned u, bool ok) {
            hist_add(sh, (u >> 8) & 0xFFFu, ok && (u & 0xFFF00000u) == prefix);
        });
    }
    if (pass_done(rv, collect ? nullptr : sh, &s_last)) {
        if (collect) {
            if (threadIdx.x == 0) {
                rv.ctrl->state = kStateSelect;
                rv.ctrl->ticket = 0u;
            }
        } else {
            pick_bucket(rv, kBins, s_need, s_scan, &s_pick);
            if (threadIdx.x == 0) {
                rv.ctrl->prefix = prefix | (s_pick.digit << 8);
                rv.ctrl->need = s_need - s_pick.above;
            }
        }
    }
}

// Exact pass 3 (only after a histogram pass 2): collect the keys above the
// 24-bit prefix, histogram the low 8 bits of the keys in it.  The last block
// fixes the k-th key T and appends the keys in (T, prefix | 0xFF], which the
// histogram gives value by value.  Fewer than k keys are above T, so the
// buffer (cap >= k) holds them all.
__global__ void __launch_bounds__(kRThreads, 2)
radix_exact3_kernel(const int32_t* __restrict__ in, size_t n, unsigned char* __restrict__ scratch, unsigned cap) {
    __shared__ unsigned sh[kBins];
    __shared__ unsigned stage[kRThreads / 32][64];
    __shared__ unsigned long long s_scan[64];
    __shared__ Bucket s_pick;
    __shared__ unsigned s_cnt[256], s_off[256];
    __shared__ int s_last, s_go;
    __shared__ unsigned s_prefix, s_need;
    const RadixView rv = radix_view(scratch);
    if (threadIdx.x == 0) {
        s_go = __ldcg(&rv.ctrl->state) == kStateExact;
        s_prefix = __ldcg(&rv.ctrl->prefix);
        s_need = __ldcg(&rv.ctrl->need);
    }
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
    if (!s_go) return;
    const unsigned prefix = s_prefix;
    WarpAppender ap{stage[threadIdx.x >> 5], 0u, false};
    for_each_key(in, n, [&](unsigned u, bool ok) {
        ap.push(rv, cap, u, ok && u > (prefix | 0xFFu));
        hist_add(sh, u & 0xFFu, ok && (u & 0xFFFFFF00u) == prefix);
    });
    ap.flush(rv, cap);
    if (pass_done(rv, sh, &s_last)) {
        // Bin counts, read before pick_bucket clears them.  Bins above the
        // k-th key's hold fewer than k keys in all.
        if (threadIdx.x < 256) s_cnt[threadIdx.x] = (unsigned)min(__ldcg(&rv.hist[threadIdx.x]), 0xFFFFFFFFull);
        pick_bucket(rv, 256, s_need, s_scan, &s_pick);
        const unsigned d = s_pick.digit;
        const unsigned nb = (unsigned)__ldcg(&rv.ctrl->nbuf);
        if (threadIdx.x == 0) {
            unsigned acc = 0;
            for (unsigned e = d + 1; e < 256; ++e) {
                s_off[e] = acc;
                acc += s_cnt[e];
            }
        }
        __syncthreads();
        for (unsigned e = d + 1; e < 256; ++e)
            for (unsigned i = threadIdx.x; i < s_cnt[e]; i += blockDim.x) rv.buf[nb + s_off[e] + i] = prefix | e;
        if (threadIdx.x == 0) {
            rv.ctrl->t = prefix | d;
            rv.ctrl->nbuf = (unsigned long long)nb + s_pick.above;
            rv.ctrl->state = kStateSorted;
        }
    }
}

// ---------------------------------------------------------------------------
// Cluster kernel: select in 8 CTAs' shared memory, then plan the sort.

__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives and waits; release and
// acquire order shared and global memory across the cluster.
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The word, or the 16-byte-aligned four words, at p's offset in the shared
// memory of the cluster's CTA `rank`.
__device__ __forceinline__ unsigned cluster_addr(const unsigned* p, unsigned rank) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(p);
    unsigned ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    return ra;
}
__device__ __forceinline__ unsigned ld_cluster(const unsigned* p, unsigned rank) {
    unsigned v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr(p, rank)) : "memory");
    return v;
}
__device__ __forceinline__ uint4 ld_cluster_v4(const unsigned* p, unsigned rank) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(cluster_addr(p, rank))
                 : "memory");
    return v;
}

enum : int { kClFull = 0, kClSample = 1, kClFinal = 2 };

constexpr int kMaxRanges = 128;        // sort ranges (one sort CTA each)
constexpr unsigned kRangeKeys = 768;   // keys a sort range aims at
constexpr unsigned kMaxPlanned = 48;   // ranges planned from the sample (heavy values add more)
constexpr unsigned kPlanSamples = 256; // splitter sample, at most
constexpr int kSortThreads = 1024;
constexpr int kSortCap = kRadixMaxK;   // keys one sort CTA holds: a range has fewer than k

// What the cluster leaves for the sort kernel (at kRadixCandOffset).
struct RadixPlan {
    unsigned nranges;           // ranges to sort (0: no key above the k-th)
    unsigned seg_off[kClCtas];  // keys above the k-th: buf[seg_off[r] .. + seg_cnt[r]) per CTA r
    unsigned seg_cnt[kClCtas];
    unsigned lb[kMaxRanges];    // range q: keys u with lb[q] <= u < lb[q-1] (range 0: u >= lb[0])
};
static_assert(sizeof(RadixPlan) <= kRadixPlanBytes, "plan area");

struct ClSmem {
    unsigned keys[kClSlice];              // the CTA's keys, then the ones above the k-th
    unsigned hist[2][256];                // digit histograms (read by the other CTAs)
    unsigned samp[kPlanSamples];          // rank 0: the gathered sample, sorted
    unsigned mysamp[kPlanSamples];        // this CTA's part of it (read by rank 0)
    unsigned ccount[kClCtas];             // every CTA's count of keys above the k-th
    unsigned wcnt[kClWarps];
    unsigned woff[kClWarps];
    unsigned lb[kMaxRanges];              // rank 0: the range table being built
    unsigned mine_count;                  // this CTA's count (read by rank 0)
    unsigned pick_digit;
    unsigned pick_above;
};

// mode kClFull:   select among the n input values (n <= cap) and plan the
//                 sort of the TopK.
// mode kClSample: select the j-th largest of 2^18 sampled keys; write it to
//                 the control words as the filter threshold.
// mode kClFinal:  select among the buffered keys as the control words say,
//                 plan the sort and zero the control words.
// In the first and last modes the copies of the k-th key are written here;
// the keys above it are left, per CTA, in the buffer for the sort kernel.
__global__ void __cluster_dims__(kClCtas, 1, 1) __launch_bounds__(kClThreads, 1)
radix_cluster_kernel(const int32_t* __restrict__ in, size_t n, int k, unsigned j_sample, int32_t* __restrict__ out,
                     unsigned char* __restrict__ scratch, unsigned cap, int mode) {
    extern __shared__ __align__(16) unsigned char radix_cl_smem[];
    ClSmem& S = *reinterpret_cast<ClSmem*>(radix_cl_smem);
    const RadixView rv = radix_view(scratch);
    const unsigned rank = cluster_rank();
    const unsigned tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

    // What this launch selects from: C keys; the j-th largest (select), or
    // all of them above a known T.
    unsigned C, j = 0, T = 0;
    bool select = true;
    if (mode == kClFull) {
        C = (unsigned)n;
        j = (unsigned)k;
    } else if (mode == kClSample) {
        C = (unsigned)kRadixClusterCap;
        j = j_sample;
    } else {
        // The earlier launches leave Select (nbuf >= k keys, at most cap) or
        // Sorted (fewer than k keys, all above t); anything else would be a
        // broken pipeline, and then nothing is read from the buffer.
        const unsigned st = __ldcg(&rv.ctrl->state);
        const unsigned long long nb = __ldcg(&rv.ctrl->nbuf);
        C = (unsigned)min(nb, (unsigned long long)cap);
        if (st == kStateSelect && C >= (unsigned)k) {
            j = (unsigned)k;
        } else {
            select = false;
            T = __ldcg(&rv.ctrl->t);
            if (st != kStateSorted || C >= (unsigned)k) C = 0;
        }
    }
    const unsigned per = (C + kClCtas - 1) / kClCtas;
    const unsigned lo = min(C, rank * per);
    const unsigned mine = min(C, lo + per) - lo;

    // Load the CTA's slice, 16 loads in flight per thread (indices past the
    // slice load its last key again and are not stored).
    constexpr int kLd = 16;
    for (unsigned base = 0; base < mine; base += kLd * kClThreads) {
        unsigned v[kLd];
        if (mode == kClFinal) {
#pragma unroll
            for (int u = 0; u < kLd; ++u) v[u] = __ldcg(rv.buf + lo + min(base + u * kClThreads + tid, mine - 1));
        } else if (mode == kClFull) {
#pragma unroll
            for (int u = 0; u < kLd; ++u) v[u] = key_of(__ldg(in + lo + min(base + u * kClThreads + tid, mine - 1)));
        } else {
#pragma unroll
            for (int u = 0; u < kLd; ++u) {
                const unsigned x = lo + min(base + u * kClThreads + tid, mine - 1);
                const size_t pos = (size_t)(x / kSegLen) * (n - kSegLen) / (kSegments - 1) + (x % kSegLen);
                v[u] = key_of(__ldg(in + pos));
            }
        }
#pragma unroll
        for (int u = 0; u < kLd; ++u) {
            const unsigned i = base + u * kClThreads + tid;
            if (i < mine) S.keys[i] = v[u];
        }
    }
    __syncthreads();

    // Warp w owns the run S.keys[w0 .. w0 + cnt) of its 1024-key sub-slice;
    // each pass below compacts the run in place (order kept).
    const unsigned w0 = w * 1024u;
    unsigned cnt = mine > w0 ? min(1024u, mine - w0) : 0u;

    // Select: four 8-bit digit levels.  Each level drops the keys below the
    // bucket chosen so far (keys above it stay: they are in the answer) and
    // histograms the next digit of the keys in it; the 256-bin histogram is
    // summed over the cluster's CTAs by one warp (16-byte remote loads), and
    // every CTA finds the same bucket.
    unsigned need;
    if (select) {
        unsigned prefix = 0;
        need = j;
        for (int level = 0; level < 4; ++level) {
            const int shift = 24 - 8 * level;
            const unsigned fixed = level == 0 ? 0u : (0xFFFFFFFFu << (32 - 8 * level));
            unsigned* H = S.hist[level & 1];
            if (tid < 256) H[tid] = 0u;
            __syncthreads();
            unsigned kept = 0;
            for (unsigned m = 0; m < cnt; m += 32) {
                const unsigned i = m + lane;
                const bool valid = i < cnt;
                const unsigned u = valid ? S.keys[w0 + i] : 0u;
                hist_add(H, (u >> shift) & 0xFFu, valid && (u & fixed) == prefix);
                const bool keep = valid && (u & fixed) >= prefix;
                const unsigned b = __ballot_sync(kFullMask, keep);
                if (keep) S.keys[w0 + kept + __popc(b & lanemask_lt())] = u;
                kept += __popc(b);
            }
            cnt = kept;
            cluster_barrier();
            if (w == 0) {
                unsigned c[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
                for (unsigned r = 0; r < (unsigned)kClCtas; ++r) {
                    const uint4 a = ld_cluster_v4(&H[lane * 8], r);
                    const uint4 b = ld_cluster_v4(&H[lane * 8 + 4], r);
                    c[0] += a.x, c[1] += a.y, c[2] += a.z, c[3] += a.w;
                    c[4] += b.x, c[5] += b.y, c[6] += b.z, c[7] += b.w;
                }
                unsigned tot = 0;
#pragma unroll
                for (int b = 0; b < 8; ++b) tot += c[b];
                unsigned x = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_down_sync(kFullMask, x, o);
                    if ((int)lane + o < 32) x += y;
                }
                const unsigned above = x - tot;
                if (above < need && need <= above + tot) {
                    unsigned acc = above;
#pragma unroll
                    for (int b = 7; b >= 0; --b) {
                        if (acc + c[b] >= need) {
                            S.pick_digit = lane * 8 + b;
                            S.pick_above = acc;
                            break;
                        }
                        acc += c[b];
                    }
                }
            }
            __syncthreads();
            prefix |= S.pick_digit << shift;
            need -= S.pick_above;
            __syncthreads();
        }
        T = prefix;
    } else {
        need = (unsigned)k - C;
    }

    if (mode == kClSample) {
        if (rank == 0 && tid == 0) rv.ctrl->t = T;
        cluster_barrier();  // keep this CTA's shared memory until every CTA has read it
        return;
    }

    // Keys above T: compact the runs once more, then the CTA's survivors go
    // out contiguously to its own part of the buffer.
    unsigned cw = 0;
    for (unsigned m = 0; m < cnt; m += 32) {
        const unsigned i = m + lane;
        const unsigned u = i < cnt ? S.keys[w0 + i] : 0u;
        const bool p = i < cnt && u > T;
        const unsigned b = __ballot_sync(kFullMask, p);
        if (p) S.keys[w0 + cw + __popc(b & lanemask_lt())] = u;
        cw += __popc(b);
    }
    if (lane == 0) S.wcnt[w] = cw;
    __syncthreads();
    if (w == 0) {
        const unsigned v = S.wcnt[lane];
        unsigned x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(kFullMask, x, o);
            if ((int)lane >= o) x += y;
        }
        S.woff[lane] = x - v;
        if (lane == 31) S.mine_count = x;
    }
    __syncthreads();
    unsigned* X = rv.buf + lo;
    for (unsigned i = lane; i < cw; i += 32) X[S.woff[w] + i] = S.keys[w0 + i];
    __threadfence();
    cluster_barrier();  // every CTA's survivors and their count are out

    // Sample for the sort plan.
    if (tid < (unsigned)kClCtas) S.ccount[tid] = ld_cluster(&S.mine_count, tid);
    __syncthreads();
    unsigned total = 0;
#pragma unroll
    for (int r = 0; r < kClCtas; ++r) total += S.ccount[r];
    // About kPlanSamples in all (never more): a CTA's share of them follows
    // its share of the keys above T.
    auto samples_of = [&](unsigned c) -> unsigned {
        return total ? (unsigned)(((unsigned long long)c * kPlanSamples) / total) : 0u;
    };
    {
        const unsigned my_c = S.mine_count, my_s = samples_of(my_c);
        for (unsigned i = tid; i < my_s; i += kClThreads) S.mysamp[i] = X[(unsigned long long)i * my_c / my_s];
    }
    cluster_barrier();  // samples out
    unsigned ns = 0;
    if (rank == 0 && total) {
        unsigned soff[kClCtas + 1];
#pragma unroll
        for (int r = 0; r < kClCtas; ++r) {
            soff[r] = ns;
            ns += samples_of(S.ccount[r]);
        }
        soff[kClCtas] = ns;
        for (unsigned i = tid; i < kPlanSamples; i += kClThreads) {
            unsigned v = 0u;
            if (i < ns) {
                unsigned r = 0;
                while (r + 1 < (unsigned)kClCtas && soff[r + 1] <= i) ++r;
                v = ld_cluster(&S.mysamp[i - soff[r]], r);
            }
            S.samp[i] = v;
        }
    }
    cluster_barrier();  // rank 0 has read every sample; no remote reads after this

    if (rank == 0) {
        RadixPlan* plan = reinterpret_cast<RadixPlan*>(scratch + kRadixCandOffset);
        if (tid < (unsigned)kClCtas) {
            plan->seg_off[tid] = min(C, tid * per);
            plan->seg_cnt[tid] = S.ccount[tid];
        }
        if (w == 0) {
            // One warp plans the ranges: R - 1 splitters at even positions of
            // the sorted sample, about kRangeKeys keys apart; a splitter value
            // that repeats at a neighbouring position (a value holding a
            // range's worth of keys) also bounds a range holding only that
            // value, which needs no sorting.  The last range ends at T + 1.
            unsigned nr = 0;
            if (total) {
                unsigned v[kPlanSamples / 32];
#pragma unroll
                for (int jj = 0; jj < (int)(kPlanSamples / 32); ++jj) v[jj] = S.samp[jj * 32 + lane];
                warp_sort_desc(v, (int)lane);
#pragma unroll
                for (int jj = 0; jj < (int)(kPlanSamples / 32); ++jj) S.samp[jj * 32 + lane] = v[jj];
                __syncwarp();
                const unsigned R = min(kMaxPlanned, max(1u, (total + kRangeKeys - 1) / kRangeKeys));
                unsigned bnd[4] = {0u, 0u, 0u, 0u};  // candidate bounds at positions jj * 32 + lane; 0 = none
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const unsigned q = lane + 1 + 32 * h;  // splitter q of 1 .. R-1
                    if (q < R) {
                        const unsigned c = S.samp[q * ns / R];
                        const bool dup = (q >= 2 && S.samp[(q - 1) * ns / R] == c) ||
                                         (q + 1 < R && S.samp[(q + 1) * ns / R] == c);
                        bnd[2 * h] = c;
                        bnd[2 * h + 1] = (dup && c != 0xFFFFFFFFu) ? c + 1 : 0u;
                    }
                }
                if (lane == 31) bnd[3] = T + 1;  // position 127: no splitter lands there (R <= 48)
                warp_sort_desc(bnd, (int)lane);
                // Keep the distinct nonzero bounds, in descending order.
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const unsigned prev_in_warp = __shfl_up_sync(kFullMask, bnd[jj], 1);
                    const unsigned prev_last = __shfl_sync(kFullMask, jj ? bnd[jj - 1] : 0u, 31);
                    const unsigned prev = lane ? prev_in_warp : (jj ? prev_last : 0xFFFFFFFFu);
                    const bool keep = bnd[jj] != 0u && (bnd[jj] != prev || (jj == 0 && lane == 0));
                    const unsigned b = __ballot_sync(kFullMask, keep);
                    if (keep) S.lb[nr + __popc(b & lanemask_lt())] = bnd[jj];
                    nr += __popc(b);
                }
                __syncwarp();
                for (unsigned i = lane; i < nr; i += 32) plan->lb[i] = S.lb[i];
            }
            if (lane == 0) plan->nranges = nr;
        }
    }
    // Copies of the k-th key fill the rest.
    for (unsigned i = total + rank * kClThreads + tid; i < (unsigned)k; i += kClCtas * kClThreads)
        out[i] = value_of(T);
    if (mode == kClFinal && rank == 0 && tid < (unsigned)kCtrlWords) reinterpret_cast<unsigned*>(rv.ctrl)[tid] = 0u;
}

// Sort kernel: CTA q sorts range q of the plan.  It reads every key above
// the k-th (fewer than k, from L2), counts those in higher ranges for its
// output offset, and sorts its own in shared memory; a single-value range
// is only counted and written.
__global__ void __launch_bounds__(kSortThreads, 1)
radix_sort_kernel(int32_t* __restrict__ out, const unsigned char* __restrict__ scratch) {
    extern __shared__ __align__(16) unsigned radix_sort_smem[];
    __shared__ unsigned s_fill;
    __shared__ unsigned s_red[2][32];
    const RadixPlan* plan = reinterpret_cast<const RadixPlan*>(scratch + kRadixCandOffset);
    const unsigned* buf = reinterpret_cast<const unsigned*>(scratch + kRadixBufOffset);
    const unsigned q = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (q >= __ldcg(&plan->nranges)) return;
    const unsigned lb = __ldcg(&plan->lb[q]);
    const bool has_ub = q > 0;
    const unsigned ub = has_ub ? __ldcg(&plan->lb[q - 1]) : 0u;
    const bool single = has_ub ? ub == lb + 1 : lb == 0xFFFFFFFFu;
    if (tid == 0) s_fill = 0u;
    __syncthreads();
    // The keys above the k-th, as one index space over the CTAs' parts.
    unsigned seg_off[kClCtas], seg_start[kClCtas], total = 0;
#pragma unroll
    for (int r = 0; r < kClCtas; ++r) {
        seg_off[r] = __ldcg(&plan->seg_off[r]);
        seg_start[r] = total;
        total += __ldcg(&plan->seg_cnt[r]);
    }
    unsigned above = 0, inr = 0;
    constexpr int kLd = 8;
    for (unsigned base = 0; base < total; base += kLd * kSortThreads) {
        unsigned v[kLd];
#pragma unroll
        for (int u = 0; u < kLd; ++u) {
            const unsigned g = min(base + u * kSortThreads + tid, total - 1);
            unsigned off = seg_off[0] + g;
#pragma unroll
            for (int r = 1; r < kClCtas; ++r)
                if (g >= seg_start[r]) off = seg_off[r] + (g - seg_start[r]);
            v[u] = __ldcg(buf + off);
        }
#pragma unroll
        for (int u = 0; u < kLd; ++u) {
            const bool ok = base + u * kSortThreads + tid < total;
            above += (ok && has_ub && v[u] >= ub) ? 1u : 0u;
            const bool p = ok && v[u] >= lb && (!has_ub || v[u] < ub);
            inr += p ? 1u : 0u;
            if (!single) {
                const unsigned b = __ballot_sync(kFullMask, p);
                if (b) {
                    const int leader = __ffs(b) - 1;
                    unsigned pos = 0;
                    if ((int)lane == leader) pos = atomicAdd(&s_fill, (unsigned)__popc(b));
                    pos = __shfl_sync(kFullMask, pos, leader);
                    if (p) radix_sort_smem[pos + __popc(b & lanemask_lt())] = v[u];
                }
            }
        }
    }
    above = __reduce_add_sync(kFullMask, above);
    inr = __reduce_add_sync(kFullMask, inr);
    if (lane == 0) {
        s_red[0][w] = above;
        s_red[1][w] = inr;
    }
    __syncthreads();
    above = 0;
    inr = 0;
#pragma unroll
    for (int i = 0; i < kSortThreads / 32; ++i) {
        above += s_red[0][i];
        inr += s_red[1][i];
    }
    if (single) {
        for (unsigned i = tid; i < inr; i += kSortThreads) out[above + i] = value_of(lb);
        return;
    }
    const int L = next_pow2((int)max(inr, 2u));
    for (unsigned i = inr + tid; i < (unsigned)L; i += kSortThreads) radix_sort_smem[i] = 0u;
    block_sort_smem_desc(radix_sort_smem, L);
    for (unsigned i = tid; i < inr; i += kSortThreads) out[above + i] = value_of(radix_sort_smem[i]);
}

struct RadixFit {
    int grid = 0;  // persistent grid of the grid passes
};

cudaError_t radix_fit(int device, RadixFit* out) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static RadixFit cache[kMaxDev];
    if (device < 0 || device >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[device].grid == 0) {
        int sms = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        if (e != cudaSuccess) return e;
        const void* passes[] = {reinterpret_cast<const void*>(&radix_filter_kernel),
                                reinterpret_cast<const void*>(&radix_exact1_kernel),
                                reinterpret_cast<const void*>(&radix_exact2_kernel),
                                reinterpret_cast<const void*>(&radix_exact3_kernel)};
        int per_sm = 1 << 30;
        for (const void* f : passes) {
            int b = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, f, kRThreads, 0);
            if (e != cudaSuccess) return e;
            if (b < per_sm) per_sm = b;
        }
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&radix_cluster_kernel),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(ClSmem));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&radix_sort_kernel),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kSortCap * sizeof(unsigned)));
        if (e != cudaSuccess) return e;
        cache[device].grid = sms * (per_sm < 1 ? 1 : per_sm);
    }
    *out = cache[device];
    return cudaSuccess;
}

}  // namespace

cudaError_t radix_launch(cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out, void* scratch,
                         size_t cap, int* launches) {
    *launches = 0;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    RadixFit f;
    e = radix_fit(device, &f);
    if (e != cudaSuccess) return e;
    if (cap > kRadixClusterCap) cap = kRadixClusterCap;
    const int opt_cap = radix_cap_option();
    if (opt_cap > 0 && (size_t)opt_cap < cap) cap = (size_t)opt_cap;
    if (cap < (size_t)k) cap = (size_t)k;
    auto* sc = static_cast<unsigned char*>(scratch);
    const unsigned ucap = (unsigned)cap;
    const size_t cl_smem = sizeof(ClSmem), sort_smem = kSortCap * sizeof(unsigned);
    if (n <= cap) {
        radix_cluster_kernel<<<kClCtas, kClThreads, cl_smem, s>>>(in, n, k, 0u, out, sc, ucap, kClFull);
        radix_sort_kernel<<<kMaxRanges, kSortThreads, sort_smem, s>>>(out, sc);
        *launches = 2;
        return cudaGetLastError();
    }
    // Sample rank: k's expected share of the sample plus four standard
    // deviations and a floor of 16, so that at least k keys are >= t.
    const double lam = (double)k * (double)kRadixClusterCap / (double)n;
    const double jd = std::ceil(lam + 4.0 * std::sqrt(lam) + 16.0);
    unsigned j = jd >= (double)kRadixClusterCap ? (unsigned)kRadixClusterCap : (unsigned)jd;
    const int opt_j = radix_sample_rank_option();
    if (opt_j > 0) j = (size_t)opt_j < kRadixClusterCap ? (unsigned)opt_j : (unsigned)kRadixClusterCap;
    const size_t per_block = (size_t)kRThreads * kRU * 4;
    size_t grid = (n + per_block - 1) / per_block;
    if (grid > (size_t)f.grid) grid = f.grid;
    if (grid < 1) grid = 1;
    radix_cluster_kernel<<<kClCtas, kClThreads, cl_smem, s>>>(in, n, k, j, out, sc, ucap, kClSample);
    radix_filter_kernel<<<(int)grid, kRThreads, 0, s>>>(in, n, k, sc, ucap);
    radix_exact1_kernel<<<(int)grid, kRThreads, 0, s>>>(in, n, k, sc, ucap);
    radix_exact2_kernel<<<(int)grid, kRThreads, 0, s>>>(in, n, sc, ucap);
    radix_exact3_kernel<<<(int)grid, kRThreads, 0, s>>>(in, n, sc, ucap);
    radix_cluster_kernel<<<kClCtas, kClThreads, cl_smem, s>>>(in, n, k, 0u, out, sc, ucap, kClFinal);
    radix_sort_kernel<<<kMaxRanges, kSortThreads, sort_smem, s>>>(out, sc);
    *launches = 7;
    return cudaGetLastError();
}

}  // namespace topk
