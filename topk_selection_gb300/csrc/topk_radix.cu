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
//   sample   one cluster of 8 CTAs gathers 2^16 keys from 4096 evenly
//            spaced 16-element segments and selects the j-th largest, j a few
//            standard deviations above k's expected share of the sample.
//            That key is the filter threshold t.
//   filter   a persistent grid reads the input once: keys above t go to the
//            candidate buffer, keys equal to t are counted.  The last block
//            to finish decides what follows:
//              buffer count >= k and it fits   -> select the k-th in the buffer
//              buffer + equal count >= k       -> t is the k-th key
//              otherwise                       -> the exact passes
//   exact    one grid launch that does work only when the sample misled the
//            filter (otherwise every block reads the state word and
//            returns); its three passes, separated by in-kernel gates:
//              pass 1   12-bit histogram of the top bits -> bucket b1
//              pass 2   if every key at or above b1 fits the buffer, collect
//                       them (then select in the buffer); else histogram the
//                       next 12 bits of the keys in b1 -> bucket b2
//              pass 3   collect the keys above the 24-bit prefix and
//                       histogram the low 8 bits of the keys in it; that
//                       fixes the k-th key T, and the keys between T and the
//                       prefix's top are written from the histogram
//   final    when k <= kSmallCap and the buffer fits one CTA's shared memory
//            (the usual case for such k), one CTA selects the k-th key T with
//            8-bit digit histograms and sorts the keys above it.  Else one
//            cluster loads the buffer into its 8 CTAs' shared memory and
//            selects T with cluster-wide 8-bit digit histograms (summed
//            through distributed shared memory).  The digits start below
//            the bits that every key in the buffer shares.  At most kSmallCap keys
//            above T: rank 0 gathers and sorts them all.
//            Otherwise their value range is cut into ranges of about 256
//            keys -- from a cluster-wide histogram of the 10 bits below the
//            common prefix of [T + 1, max], or, when one bucket is too dense,
//            from a splitter sample weighted by each CTA's share (a value
//            that dominates the sample gets a range of its own).  Every CTA
//            counts its keys per range, writes them straight to their range
//            of the output, and each range is then sorted in place by one
//            warp.  Copies of the k-th key fill the rest of the output.
// When n fits one cluster, the cluster kernel alone runs, on the input itself.
// Every decision stays on the device, so a call only enqueues work.  The
// exact passes' blocks wait for one another at their gates with a bounded
// poll; every other wait in these kernels is a hardware barrier
// (__syncthreads, the cluster barrier), so none can hang.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "topk_device.cuh"
#include "topk_internal.h"
#include "topk_sortnet.cuh"

namespace topk {

namespace {

constexpr int kRThreads = 512;  // grid passes
constexpr int kRU = 8;          // 16-byte loads in flight per thread
constexpr int kFilterPrefetch = 6;  // batches per block fetched into L2 while the sample runs
constexpr int kBins = 4096;     // 12-bit digits

constexpr int kClCtas = 8;  // CTAs per cluster (portable size)
constexpr int kClThreads = 1024;
constexpr int kClWarps = kClThreads / 32;
constexpr int kClSlice = 32768;  // keys per CTA
constexpr unsigned kSegLen = 16;
// The threshold sample: 2^16 keys (a quarter of what a cluster holds)
// still put the filter's expected candidates far below the buffer (about
// j * n / 2^16 for the sample rank j below), at a quarter of the loads.
constexpr unsigned kSampleKeys = 1u << 16;
constexpr unsigned kSegments = kSampleKeys / kSegLen;
constexpr int kSampleVec = (int)(kSampleKeys / (4u * kClCtas * kClThreads));  // 16-byte loads per thread
static_assert(kSampleVec >= 1 && kSampleVec * 4 * kClCtas * kClThreads == (int)kSampleKeys, "sample split");
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
    unsigned gate;            // exact passes: the last pass whose bucket is picked
    unsigned pad[53];
};
static_assert(sizeof(RadixCtrl) == 256, "one line");
constexpr int kCtrlWords = 11;

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

// Fetch `bytes` (a multiple of 16; src 16-byte aligned) of global memory
// into L2, asynchronously; nothing waits for it.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
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
template <int KIND, class FV, class FT>
__device__ __forceinline__ void for_each_vec(const int32_t* __restrict__ in, size_t n, FV f_vec, FT f_tail) {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(in);
    size_t head = ((16u - (unsigned)(addr & 15u)) & 15u) >> 2;
    if (head > n) head = n;
    const int4* body = reinterpret_cast<const int4*>(in + head);
    const size_t nvec = (n - head) >> 2;
    const size_t tail0 = head + nvec * 4;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const uint64_t policy = l2_evict_first_policy();  // the input is read once per pass
    for (size_t base = (size_t)blockIdx.x * blockDim.x * kRU; base < nvec; base += stride * kRU) {
        int4 r[kRU];
#pragma unroll
        for (int u = 0; u < kRU; ++u) {
            const size_t i = base + (size_t)u * blockDim.x + threadIdx.x;
            r[u] = i < nvec ? ld_nc_hint(body + i, policy) : make_int4(0, 0, 0, 0);
        }
        // The key map after all kRU loads are out, so that none waits for another.
#pragma unroll
        for (int u = 0; u < kRU; ++u) f_vec(ordered4<KIND>(r[u]), base + (size_t)u * blockDim.x + threadIdx.x < nvec);
    }
    if (blockIdx.x == 0 && threadIdx.x < 32) {
        const size_t ns = head + (n - tail0);
        const size_t lane = threadIdx.x;
        const size_t pos = lane < head ? lane : tail0 + (lane - head);
        f_tail(lane < ns ? ordered<KIND>(in[pos]) : 0, lane < ns);
    }
}

template <int KIND, class F>
__device__ __forceinline__ void for_each_key(const int32_t* __restrict__ in, size_t n, F f) {
    for_each_vec<KIND>(
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
template <int KIND>
__global__ void __launch_bounds__(kRThreads, 2)
radix_filter_kernel(const int32_t* __restrict__ in, size_t n, int k, unsigned char* __restrict__ scratch,
                    unsigned cap) {
    __shared__ unsigned stage[kRThreads / 32][64];
    __shared__ unsigned long long s_neq;
    __shared__ int s_last;
    // The input is final before this kernel starts: it is launched only
    // once every CTA of the sample has passed its own wait for the work
    // before the plan.  Only the threshold comes from the sample.  So while
    // the sample runs, each block fetches its first kFilterPrefetch batches
    // of the input into L2 (the batches for_each_vec reads first).
    if (threadIdx.x == 0) {
        const uintptr_t addr = reinterpret_cast<uintptr_t>(in);
        size_t head = ((16u - (unsigned)(addr & 15u)) & 15u) >> 2;
        if (head > n) head = n;
        const int4* body = reinterpret_cast<const int4*>(in + head);
        const size_t nvec = (n - head) >> 2, batch = (size_t)blockDim.x * kRU;
        for (int p = 0; p < kFilterPrefetch; ++p) {
            const size_t v0 = (size_t)blockIdx.x * batch + (size_t)p * gridDim.x * batch;
            if (v0 >= nvec) break;
            const size_t nv = nvec - v0 < batch ? nvec - v0 : batch;
            prefetch_l2(body + v0, (uint32_t)(nv * 16));
        }
    }
    grid_dependency_wait();  // launched early (launch_pdl): wait for the previous kernel's writes
    launch_dependents();
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
    for_each_vec<KIND>(
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

// Exact passes, one launch.  When the sample did not mislead the filter
// (the usual case) every block reads the state word and returns.  Else:
//   pass 1   12-bit histogram of the top bits -> bucket b1
//   pass 2   if every key at or above b1 fits the buffer, collect them (then
//            select in the buffer); else histogram the next 12 bits of the
//            keys in b1 -> bucket b2
//   pass 3   (after a histogram pass 2) collect the keys above the 24-bit
//            prefix and histogram the low 8 bits of the keys in it; the last
//            block fixes the k-th key T and appends the keys in
//            (T, prefix | 0xFF] from the histogram, value by value.
// The last block of a pass picks the bucket and opens the pass's gate (a
// control word); the others wait for it, polling with a bound.  The grid is
// at most what the SMs hold at once, and the next kernel of the plan is
// released only when the passes end, so every block of the grid is, or
// becomes, resident while the others wait.  A wait that runs out sets the
// status word and goes on (the result is then invalid; every buffer write
// stays inside the buffer).
__device__ __forceinline__ void exact_gate_open(const RadixView& rv, unsigned pass) {
    __threadfence();
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&rv.ctrl->gate), "r"(pass) : "memory");
}
__device__ void exact_gate_wait(const RadixView& rv, unsigned pass, unsigned* status) {
    if (threadIdx.x == 0) {
        unsigned g = 0;
        for (int i = 0; i < kWaitSpins; ++i) {
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(g) : "l"(&rv.ctrl->gate) : "memory");
            if (g >= pass) break;
            __nanosleep(64);
        }
        if (g < pass) atomicOr(status, kStatusWaitTimeout);
    }
    __syncthreads();
}

template <int KIND>
__global__ void __launch_bounds__(kRThreads, 2)
radix_exact_kernel(const int32_t* __restrict__ in, size_t n, int k, unsigned char* __restrict__ scratch,
                   unsigned cap) {
    __shared__ unsigned sh[kBins];
    __shared__ unsigned stage[kRThreads / 32][64];
    __shared__ unsigned long long s_scan[64];
    __shared__ Bucket s_pick;
    __shared__ unsigned s_cnt[256], s_off[256];
    __shared__ int s_last, s_go;
    __shared__ unsigned s_prefix, s_mode, s_need;
    grid_dependency_wait();  // launched early (launch_pdl): wait for the previous kernel's writes
    const RadixView rv = radix_view(scratch);
    unsigned* status = reinterpret_cast<unsigned*>(scratch + kI32StatusOffset);
    if (threadIdx.x == 0) s_go = __ldcg(&rv.ctrl->state) == kStateExact;
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
    if (!s_go) return;  // (returning releases the next kernel)

    // Pass 1.
    for_each_key<KIND>(in, n, [&](unsigned u, bool ok) { hist_add(sh, u >> 20, ok); });
    if (pass_done(rv, sh, &s_last)) {
        pick_bucket(rv, kBins, (unsigned)k, s_scan, &s_pick);
        if (threadIdx.x == 0) {
            rv.ctrl->prefix = s_pick.digit << 20;
            rv.ctrl->need = (unsigned)k - s_pick.above;
            rv.ctrl->exact_mode = s_pick.above + s_pick.count <= cap ? kExactCollectAll : kExactHistogram;
            rv.ctrl->nbuf = 0ull;
            rv.ctrl->neq = 0ull;
            exact_gate_open(rv, 1u);
        }
    }
    exact_gate_wait(rv, 1u, status);

    // Pass 2.
    if (threadIdx.x == 0) {
        s_prefix = __ldcg(&rv.ctrl->prefix);
        s_mode = __ldcg(&rv.ctrl->exact_mode);
        s_need = __ldcg(&rv.ctrl->need);
    }
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
    unsigned prefix = s_prefix;
    const bool collect = s_mode == kExactCollectAll;
    if (collect) {
        WarpAppender ap{stage[threadIdx.x >> 5], 0u, false};
        for_each_key<KIND>(in, n, [&](unsigned u, bool ok) { ap.push(rv, cap, u, ok && (u & 0xFFF00000u) >= prefix); });
        ap.flush(rv, cap);
    } else {
        for_each_key<KIND>(in, n, [&](unsigned u, bool ok) {
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
                exact_gate_open(rv, 2u);
            }
        }
    }
    if (collect) return;
    exact_gate_wait(rv, 2u, status);

    // Pass 3.
    if (threadIdx.x == 0) {
        s_prefix = __ldcg(&rv.ctrl->prefix);
        s_need = __ldcg(&rv.ctrl->need);
    }
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
    prefix = s_prefix;
    WarpAppender ap{stage[threadIdx.x >> 5], 0u, false};
    for_each_key<KIND>(in, n, [&](unsigned u, bool ok) {
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
            for (unsigned i = threadIdx.x; i < s_cnt[e]; i += blockDim.x)
                if ((size_t)nb + s_off[e] + i < cap) rv.buf[nb + s_off[e] + i] = prefix | e;
        if (threadIdx.x == 0) {
            rv.ctrl->t = prefix | d;
            rv.ctrl->nbuf = (unsigned long long)nb + s_pick.above;
            rv.ctrl->state = kStateSorted;
        }
    }
}

// ---------------------------------------------------------------------------
// Cluster kernel: select, partition and sort in 8 CTAs' shared memory.

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

constexpr int kMaxRanges = 256;          // output ranges (one sorting warp each)
constexpr unsigned kMaxPlanned = 128;    // ranges cut from the sample; repeated values add up to as many
constexpr unsigned kRangeKeys = 256;     // keys a range aims at
constexpr unsigned kPlanSamples = 512;   // splitter sample, at most
// At most this many keys above T: rank 0 gathers and sorts them all itself
// (measured faster than the range plan up to ~2000 keys, slower at 4096).
constexpr unsigned kSmallCap = 2048;
static_assert(kSmallCap >= 1024, "the radix range plan sums its 1024 buckets in mysmall");
static_assert(2 * kMaxPlanned <= (unsigned)kMaxRanges, "range table");
static_assert(kClCtas * kMaxRanges == 2 * kClThreads, "two (CTA, range) counts per thread");
constexpr int kSortWarps = 4;            // warps per CTA of the sort kernel
constexpr int kSortRegCap = 512;         // a warp sorts ranges up to this in registers
constexpr int kSortCap = kRadixMaxK;     // a larger range is sorted by its CTA in shared memory

// What the cluster leaves for the sort kernel (at kRadixCandOffset).
struct RadixPlan {
    unsigned nranges;
    unsigned rstart[kMaxRanges + 1];  // range q: out[rstart[q] .. rstart[q+1])
    unsigned lb[kMaxRanges];          // range q holds keys u with lb[q] <= u < lb[q-1]
};
static_assert(sizeof(RadixPlan) <= kRadixPlanBytes, "plan area");

struct ClSmem {
    unsigned keys[kClSlice];              // the CTA's keys
    unsigned hist[2][256];                // digit histograms (read by the other CTAs)
    unsigned part[kClCtas][kMaxRanges];   // the cluster's histograms of a level; later the range counts
    unsigned samp[kPlanSamples];          // rank 0: the gathered sample
    unsigned mysamp[kPlanSamples];        // this CTA's part of it (read by rank 0)
    unsigned mysmall[kSmallCap];          // few keys above T: this CTA's, packed (read by rank 0)
    unsigned lb[kMaxRanges];              // range bounds (rank 0 builds them; the others copy)
    unsigned rcnt[kMaxRanges];            // this CTA's keys per range (read by the others)
    unsigned rstart[kMaxRanges + 1];      // output offset of each range
    unsigned rpos[kMaxRanges];            // this CTA's next output slot in each range
    unsigned ccount[kClCtas];             // every CTA's count of keys above the k-th
    unsigned wcnt[kClWarps];
    unsigned woff[kClWarps];
    unsigned mine_count;                  // this CTA's count (read by the others)
    unsigned nranges;                     // (rank 0's is read by the others)
    unsigned pick_digit;
    unsigned pick_above;
    unsigned pick_cnt;                    // keys in the picked bucket
    unsigned wmax[kClWarps];              // radix range plan: per-warp maxima of the keys above T
    unsigned cmax;                        // the CTA's maximum (read by the others)
    unsigned hi_key;                      // the cluster's maximum
    unsigned plan_ok;                     // the radix plan fits (else the splitter-sample plan)
};
static_assert(kMaxRanges == 256, "a level's histogram fits a row of part");

// After the cluster barrier that completes every CTA's histogram H: sum the
// 8 histograms (warp r reads CTA r's with 16-byte remote loads) and find the
// bucket holding the need-th largest key.  Every CTA finds the same one.
__device__ __forceinline__ void cluster_pick(ClSmem& S, const unsigned* H, unsigned need) {
    const unsigned lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (w < (unsigned)kClCtas) {
        const uint4 a = ld_cluster_v4(&H[lane * 8], w);
        const uint4 b = ld_cluster_v4(&H[lane * 8 + 4], w);
        *reinterpret_cast<uint4*>(&S.part[w][lane * 8]) = a;
        *reinterpret_cast<uint4*>(&S.part[w][lane * 8 + 4]) = b;
    }
    __syncthreads();
    if (w == 0) {
        unsigned c[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int r = 0; r < kClCtas; ++r) {
            const uint4 a = *reinterpret_cast<const uint4*>(&S.part[r][lane * 8]);
            const uint4 b = *reinterpret_cast<const uint4*>(&S.part[r][lane * 8 + 4]);
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
                    S.pick_cnt = c[b];
                    break;
                }
                acc += c[b];
            }
        }
    }
    __syncthreads();
}

// The same within one CTA: H is this CTA's histogram, complete after a
// __syncthreads.
__device__ __forceinline__ void cta_pick(ClSmem& S, const unsigned* H, unsigned need) {
    const unsigned lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (w == 0) {
        unsigned c[8], tot = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            c[b] = H[lane * 8 + b];
            tot += c[b];
        }
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
                    S.pick_cnt = c[b];
                    break;
                }
                acc += c[b];
            }
        }
    }
    __syncthreads();
}

// Range of key u: the first q with u >= lb[q] (lb descending, lb[nr-1] <= u).
__device__ __forceinline__ unsigned range_of(const unsigned* lb, unsigned nr, unsigned u) {
    unsigned lo = 0, hi = nr - 1;
    while (lo < hi) {
        const unsigned mid = (lo + hi) >> 1;
        if (u >= lb[mid])
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

// mode kClFull:   the TopK of the n input values (n <= cap).
// mode kClSample: select the j-th largest of kSampleKeys sampled keys; write it to
//                 the control words as the filter threshold.
// mode kClFinal:  the TopK from the buffered keys, as the control words say;
//                 zero the control words.
template <int KIND>
__global__ void __cluster_dims__(kClCtas, 1, 1) __launch_bounds__(kClThreads, 1)
radix_cluster_kernel(const int32_t* __restrict__ in, size_t n, int k, unsigned j_sample, int32_t* __restrict__ out,
                     unsigned char* __restrict__ scratch, unsigned cap, int mode, uint32_t* __restrict__ bigk) {
    extern __shared__ __align__(16) unsigned char radix_cl_smem[];
    ClSmem& S = *reinterpret_cast<ClSmem*>(radix_cl_smem);
    grid_dependency_wait();  // launched early (launch_pdl): wait for the previous kernel's writes
    launch_dependents();
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
        C = kSampleKeys;
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
    // One CTA does the final alone when the buffer fits its shared memory
    // and the answer is small (the usual case for k <= kSmallCap).  The
    // other CTAs leave at once (after the control words are read: rank 0
    // clears them at the end), and nothing below waits on them or reads
    // their shared memory.
    const bool solo = mode == kClFinal && (unsigned)k <= kSmallCap && C <= (unsigned)kClSlice;
    if (solo) cluster_barrier();
    if (solo && rank != 0) return;
    const unsigned per = solo ? C : (C + kClCtas - 1) / kClCtas;
    const unsigned lo = solo ? 0u : min(C, rank * per);
    const unsigned mine = min(C, lo + per) - lo;

    // The keys to select from lie in [klo, 2^32 - 1]: above the filter's
    // threshold (or, after exact pass 2 collected them, at or above its
    // prefix) for the buffer, anywhere otherwise.  So they share klo's
    // bits above `top0`, and the digit levels start just below those: for a
    // small k the buffer's keys share their top 12 bits or more.
    unsigned klo = 0;
    if (mode == kClFinal && select)
        klo = __ldcg(&rv.ctrl->exact_mode) == kExactCollectAll ? __ldcg(&rv.ctrl->prefix) : __ldcg(&rv.ctrl->t) + 1u;
    const int top0 = 32 - __clz((int)~klo);  // klo's leading one bits are the common prefix
    const unsigned pre0 = top0 >= 32 ? 0u : ~((1u << top0) - 1u);
    const int sh0 = top0 > 8 ? top0 - 8 : 0;
    const unsigned dm0 = (1u << (top0 - sh0)) - 1u;

    // Load the CTA's keys, histogramming their first digit on the way (level
    // 0 of the select).
    if (tid < 256) S.hist[0][tid] = 0u;
    __syncthreads();
    if (mode == kClSample) {
        // Segment g of the sample: 16 keys from the 16-byte-aligned body,
        // four vector loads; this CTA's kSegments / 8 segments, kSampleVec
        // vectors per thread.
        const unsigned head = (unsigned)(((16u - (unsigned)(reinterpret_cast<uintptr_t>(in) & 15u)) & 15u) >> 2);
        const int4* body = reinterpret_cast<const int4*>(in + head);
        const size_t nvec = (n - head) >> 2;
        int4 v[kSampleVec];
#pragma unroll
        for (int m = 0; m < kSampleVec; ++m) {
            const unsigned x = lo / 4 + m * kClThreads + tid;
            const size_t vi = (size_t)(x >> 2) * (nvec - 4) / (kSegments - 1) + (x & 3);
            v[m] = ordered4<KIND>(__ldg(body + vi));
        }
#pragma unroll
        for (int m = 0; m < kSampleVec; ++m) {
            const uint4 u = make_uint4(key_of(v[m].x), key_of(v[m].y), key_of(v[m].z), key_of(v[m].w));
            *reinterpret_cast<uint4*>(&S.keys[(m * kClThreads + tid) * 4]) = u;
            hist_add(S.hist[0], (u.x >> sh0) & dm0, true);
            hist_add(S.hist[0], (u.y >> sh0) & dm0, true);
            hist_add(S.hist[0], (u.z >> sh0) & dm0, true);
            hist_add(S.hist[0], (u.w >> sh0) & dm0, true);
        }
    } else {
        // 16 loads in flight per thread; indices past the slice load its
        // last key again and are not stored.
        constexpr int kLd = 16;
        for (unsigned base = 0; base < mine; base += kLd * kClThreads) {
            unsigned v[kLd];
            if (mode == kClFinal) {
#pragma unroll
                for (int u = 0; u < kLd; ++u) v[u] = __ldcg(rv.buf + lo + min(base + u * kClThreads + tid, mine - 1));
            } else {
#pragma unroll
                for (int u = 0; u < kLd; ++u)
                    v[u] = key_of(ordered<KIND>(__ldg(in + lo + min(base + u * kClThreads + tid, mine - 1))));
            }
#pragma unroll
            for (int u = 0; u < kLd; ++u) {
                const unsigned i = base + u * kClThreads + tid;
                if (i < mine) S.keys[i] = v[u];
                hist_add(S.hist[0], (v[u] >> sh0) & dm0, i < mine);
            }
        }
    }
    __syncthreads();

    // Warp w owns the run S.keys[w0 .. w0 + cnt) of its 1/32 of the slice;
    // each pass below compacts the run in place (order kept).
    const unsigned share = (mine + kClWarps - 1) / kClWarps;
    const unsigned w0 = w * share;
    unsigned cnt = mine > w0 ? min(share, mine - w0) : 0u;

    // Select: digit levels of 8 bits (the last one fewer) below the common
    // prefix.  Each level after the first drops the keys below the bucket
    // chosen so far (keys above it stay: they are in the answer) and
    // histograms the next digit of the keys in it.
    if (select) {
        unsigned prefix = pre0, need = j;
        int top = top0;
        for (int level = 0; top > 0; ++level) {
            const int shift = top > 8 ? top - 8 : 0;
            const unsigned dmask = (1u << (top - shift)) - 1u;
            unsigned* H = S.hist[level & 1];
            if (level > 0) {
                const unsigned fixed = ~((1u << top) - 1u);  // top < 32 after the first level
                if (tid < 256) H[tid] = 0u;
                __syncthreads();
                unsigned kept = 0;
                for (unsigned m = 0; m < cnt; m += 32) {
                    const unsigned i = m + lane;
                    const bool valid = i < cnt;
                    const unsigned u = valid ? S.keys[w0 + i] : 0u;
                    hist_add(H, (u >> shift) & dmask, valid && (u & fixed) == prefix);
                    const bool keep = valid && (u & fixed) >= prefix;
                    const unsigned b = __ballot_sync(kFullMask, keep);
                    if (keep) S.keys[w0 + kept + __popc(b & lanemask_lt())] = u;
                    kept += __popc(b);
                }
                cnt = kept;
            }
            if (solo) {
                __syncthreads();
                cta_pick(S, H, need);
            } else {
                cluster_barrier();
                cluster_pick(S, H, need);
            }
            prefix |= S.pick_digit << shift;
            need -= S.pick_above;
            const unsigned ge = (j - need) + S.pick_cnt;  // keys at or above the bucket's lower edge
            __syncthreads();  // the pick and part are rewritten at the next level
            top = shift;
            // The sample needs only a threshold with at least j of its keys
            // above it, not its exact j-th key: once the bucket's lower edge
            // L (= prefix, lower bits zero) has between j and 2j keys at or
            // above it, L - 1 serves and the remaining levels are skipped
            // (for uniform keys, after the second level) -- as long as the
            // candidates it keeps, about ge * n / kSampleKeys, stay within
            // half the buffer.
            if (mode == kClSample && top > 0 && prefix > 0u && ge <= 2u * j &&
                (unsigned long long)ge * n <= (unsigned long long)kSampleKeys * (cap / 2u)) {
                prefix -= 1u;
                break;
            }
        }
        T = prefix;
    }

    if (mode == kClSample) {
        if (rank == 0 && tid == 0) rv.ctrl->t = T;
        cluster_barrier();  // keep this CTA's shared memory until every CTA has read it
        return;
    }

    // Keys above T, compacted in each warp's run.
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
    if (solo) {
        // Every key above T is this CTA's (fewer than k <= kSmallCap): pack,
        // sort and write them, then copies of T.
        const unsigned total = S.mine_count;
        for (unsigned m = lane; m < cw; m += 32) S.mysmall[S.woff[w] + m] = S.keys[w0 + m];
        const int P = next_pow2(total < 64 ? 64 : (int)total);
        for (unsigned i = total + tid; i < (unsigned)P; i += kClThreads) S.mysmall[i] = 0u;  // below every key > T
        __syncthreads();
        block_sort_reg_desc<unsigned, kClThreads>(S.mysmall, P);
        for (unsigned i = tid; i < total; i += kClThreads) out[i] = ordered<KIND>(value_of(S.mysmall[i]));
        for (unsigned i = total + tid; i < (unsigned)k; i += kClThreads) out[i] = ordered<KIND>(value_of(T));
        if (tid == 0) reinterpret_cast<RadixPlan*>(scratch + kRadixCandOffset)->nranges = 0u;
        if (tid < (unsigned)kCtrlWords) reinterpret_cast<unsigned*>(rv.ctrl)[tid] = 0u;
        return;
    }
    cluster_barrier();  // every CTA's count is out

    if (tid < (unsigned)kClCtas) S.ccount[tid] = ld_cluster(&S.mine_count, tid);
    __syncthreads();
    unsigned total = 0;
#pragma unroll
    for (int r = 0; r < kClCtas; ++r) total += S.ccount[r];
    unsigned nr = 0;  // ranges for the sort kernel
    if (bigk) {
        // k beyond what the range plan sorts: every CTA writes its keys
        // above T, complemented (so that an ascending sort puts the largest
        // first), to bigk[0, total) at its offset, and ~T fills [total, k);
        // the library's LSD radix sort then orders the k words.
        unsigned off = 0;
        for (unsigned r = 0; r < rank; ++r) off += S.ccount[r];
        off += S.woff[w];
        for (unsigned m = lane; m < cw; m += 32) bigk[off + m] = ~S.keys[w0 + m];
        for (unsigned i = total + rank * kClThreads + tid; i < (unsigned)k; i += kClCtas * kClThreads)
            bigk[i] = ~T;
        if (rank == 0 && tid == 0) reinterpret_cast<RadixPlan*>(scratch + kRadixCandOffset)->nranges = 0u;
        cluster_barrier();  // no CTA exits while another may read its shared memory
        if (mode == kClFinal && rank == 0 && tid < (unsigned)kCtrlWords)
            reinterpret_cast<unsigned*>(rv.ctrl)[tid] = 0u;
        return;
    }
    if (total <= kSmallCap) {
        // Few keys above T: rank 0 gathers them all, sorts them with the
        // whole CTA and writes them; the sort kernel has no ranges to do.
        // Each CTA first packs its warps' runs, in order, into mysmall.
        for (unsigned m = lane; m < cw; m += 32) S.mysmall[S.woff[w] + m] = S.keys[w0 + m];
        cluster_barrier();  // every CTA's packed keys are out
        if (rank == 0) {
            // rank 0's own keys have been packed: its key area is free.
            unsigned* all = S.keys;
            unsigned off = 0;
            for (int r = 0; r < kClCtas; ++r) {
                const unsigned c = S.ccount[r];
                for (unsigned i = tid; i < c; i += kClThreads) all[off + i] = ld_cluster(&S.mysmall[i], (unsigned)r);
                off += c;
            }
            const int P = next_pow2(total < 64 ? 64 : (int)total);
            for (unsigned i = total + tid; i < (unsigned)P; i += kClThreads) all[i] = 0u;  // below every key > T
            static_assert(kSmallCap <= 2 * kClThreads, "the register-stage sort takes two keys per thread");
            block_sort_reg_desc<unsigned, kClThreads>(all, P);
            for (unsigned i = tid; i < total; i += kClThreads) out[i] = ordered<KIND>(value_of(all[i]));
        }
    } else {
        // Radix range plan.  The keys above T lie in [lo, hi] (lo = T + 1, hi
        // their maximum) and share every bit above the highest bit where lo
        // and hi differ; the 10 bits below it cut them into at most 1024
        // buckets in key order.  Every CTA sums the cluster's bucket
        // histogram over DSMEM and builds the same range table: a range ends
        // where the exclusive count (from the top) crosses a multiple of
        // kRangeKeys, so a range holds at most kRangeKeys - 1 + its last
        // bucket's keys.  A bucket of more than kRangeKeys + 1 keys (a dense
        // value range) would overflow a warp's register sort: then the
        // splitter-sample plan runs instead.
        {
            unsigned mx = 0;
            for (unsigned m = lane; m < cw; m += 32) mx = max(mx, S.keys[w0 + m]);
            mx = __reduce_max_sync(kFullMask, mx);
            if (lane == 0) S.wmax[w] = mx;
            unsigned* hist = &S.part[0][0];  // 1024 buckets (the level histograms are done)
            hist[tid] = 0u;
            __syncthreads();
            if (w == 0) {
                const unsigned v = __reduce_max_sync(kFullMask, S.wmax[lane]);
                if (lane == 0) S.cmax = v;
            }
            __syncthreads();
            cluster_barrier();  // every CTA's maximum is out
            if (w == 0) {
                const unsigned v = lane < (unsigned)kClCtas ? ld_cluster(&S.cmax, lane) : 0u;
                const unsigned h = __reduce_max_sync(kFullMask, v);
                if (lane == 0) S.hi_key = h;
            }
            __syncthreads();
            const unsigned lo = T + 1, hi = S.hi_key;  // total > 0 keys above T: lo <= hi
            const int span = 32 - __clz((int)(lo ^ hi));  // bits below the common prefix
            const int shift = span > 10 ? span - 10 : 0;
            const unsigned base = lo >> shift, nb = (hi >> shift) - base + 1;  // nb <= 1024
            for (unsigned m = lane; m < cw; m += 32) atomicAdd(&hist[(S.keys[w0 + m] >> shift) - base], 1u);
            __syncthreads();
            cluster_barrier();  // every CTA's histogram is out
            unsigned* sum = S.mysmall;  // 1024 summed buckets
            {
                unsigned c = 0;
                if (tid < nb)
#pragma unroll 1
                    for (int r = 0; r < kClCtas; ++r) c += ld_cluster(&hist[tid], (unsigned)r);
                sum[tid] = c;
            }
            __syncthreads();
            if (w == 0) {
                // Lane l takes buckets i = 32 l .. 32 l + 31 counted from the
                // top (bucket b = nb - 1 - i).
                unsigned tot = 0, heavy = 0;
#pragma unroll 1
                for (unsigned j = 0; j < 32; ++j) {
                    const unsigned i = lane * 32 + j;
                    const unsigned c = i < nb ? sum[nb - 1 - i] : 0u;
                    tot += c;
                    heavy |= c > kRangeKeys + 1 ? 1u : 0u;
                }
                unsigned x = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(kFullMask, x, o);
                    if ((int)lane >= o) x += y;
                }
                unsigned excl = x - tot;
                unsigned nrr = 0;
#pragma unroll 1
                for (unsigned j = 0; j < 32; ++j) {
                    // Round j: lane l looks at bucket i = 32 l + j; the bounds
                    // come out in key order within each round only, so each
                    // lane first keeps its own (lanes own contiguous buckets).
                    const unsigned i = lane * 32 + j;
                    const unsigned c = i < nb ? sum[nb - 1 - i] : 0u;
                    const bool last = i < nb && (i == nb - 1 || ((excl + c) / kRangeKeys) != (excl / kRangeKeys));
                    if (last) {
                        const unsigned b = nb - 1 - i;
                        const unsigned bl = (base + b) << shift;
                        S.samp[lane * 16 + (nrr & 15)] = bl > lo ? bl : lo;  // at most 16 cuts in 32 buckets of a lane? checked below
                        ++nrr;
                    }
                    excl += c;
                }
                // A lane's 32 buckets hold at most 32 cuts; 16 slots per lane
                // suffice only when its cuts are few: otherwise the sample plan.
                const unsigned over = __reduce_or_sync(kFullMask, nrr > 16 ? 1u : 0u);
                unsigned pre = nrr;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(kFullMask, pre, o);
                    if ((int)lane >= o) pre += y;
                }
                const unsigned all_nr = __shfl_sync(kFullMask, pre, 31);
                const bool ok = !__reduce_or_sync(kFullMask, heavy) && !over && all_nr <= (unsigned)kMaxRanges;
                if (ok)
                    for (unsigned q = 0; q < nrr; ++q) S.lb[pre - nrr + q] = S.samp[lane * 16 + q];
                if (lane == 0) {
                    S.plan_ok = ok ? 1u : 0u;
                    S.nranges = ok ? all_nr : 0u;
                }
            }
            __syncthreads();
        }
        if (!S.plan_ok) {
            // Splitter sample: a CTA's share of kPlanSamples follows its share
            // of the keys above T.
            auto samples_of = [&](unsigned c) -> unsigned {
                return total ? (unsigned)(((unsigned long long)c * kPlanSamples) / total) : 0u;
            };
            {
                const unsigned my_c = S.mine_count, my_s = samples_of(my_c);
                for (unsigned i = tid; i < my_s; i += kClThreads) {
                    const unsigned g = (unsigned)((unsigned long long)i * my_c / my_s);
                    unsigned a = 0, b = kClWarps - 1;  // the last warp whose run starts at or before g
                    while (a < b) {
                        const unsigned mid = (a + b + 1) >> 1;
                        if (S.woff[mid] <= g)
                            a = mid;
                        else
                            b = mid - 1;
                    }
                    S.mysamp[i] = S.keys[a * share + (g - S.woff[a])];
                }
                // This CTA's samples, sorted descending by the whole CTA (zeros pad
                // past my_s; every sample is above T, so nonzero).  A rolled loop:
                // this runs once per launch, and an unrolled sort's straight-line
                // code would mostly wait on instruction fetch.
                const int P = next_pow2(my_s < 2 ? 2 : (int)my_s);
                for (unsigned i = my_s + tid; i < (unsigned)P; i += kClThreads) S.mysamp[i] = 0u;
                block_sort_smem_desc(S.mysamp, P);
            }
            cluster_barrier();  // sorted samples out

            if (rank == 0) {
                if (total) {
                    unsigned soff[kClCtas + 1], ns = 0;
        #pragma unroll
                    for (int r = 0; r < kClCtas; ++r) {
                        soff[r] = ns;
                        ns += samples_of(S.ccount[r]);
                    }
                    soff[kClCtas] = ns;
                    // Gather the 8 sorted lists, then merge them by rank: an element's
                    // place is its index in its own list plus, in every other list,
                    // the count of greater keys (equal keys count from lower ranks).
                    unsigned* lists = &S.part[0][0];
                    for (unsigned i = tid; i < ns; i += kClThreads) {
                        unsigned r = 0;
                        while (r + 1 < (unsigned)kClCtas && soff[r + 1] <= i) ++r;
                        lists[i] = ld_cluster(&S.mysamp[i - soff[r]], r);
                    }
                    __syncthreads();
                    for (unsigned i = tid; i < ns; i += kClThreads) {
                        unsigned r = 0;
                        while (r + 1 < (unsigned)kClCtas && soff[r + 1] <= i) ++r;
                        const unsigned v = lists[i];
                        unsigned place = i - soff[r];
                        for (unsigned o = 0; o < (unsigned)kClCtas; ++o) {
                            if (o == r) continue;
                            // first index in list o whose key is below v (o < r) or not above v (o > r)
                            unsigned a = soff[o], b = soff[o + 1];
                            while (a < b) {
                                const unsigned mid = (a + b) >> 1;
                                const unsigned x = lists[mid];
                                if (o < r ? x >= v : x > v)
                                    a = mid + 1;
                                else
                                    b = mid;
                            }
                            place += a - soff[o];
                        }
                        S.samp[place] = v;
                    }
                    __syncthreads();
                    if (w == 0) {
                        // R - 1 splitters at even positions of the sorted sample,
                        // about kRangeKeys keys apart.  A splitter value that repeats
                        // at a neighbouring position (a value holding a range's worth
                        // of keys) also bounds a range holding only that value, which
                        // needs no sorting.  The last range ends at T + 1.
                        // At least 4 samples per range keep the ranges' sizes close
                        // to their mean.
                        const unsigned R =
                            min(min(kMaxPlanned, max(1u, ns / 4)), max(1u, (total + kRangeKeys - 1) / kRangeKeys));
                        unsigned bnd[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // candidates at positions jj * 32 + lane
        #pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const unsigned q = lane + 1 + 32 * h;  // splitter q of 1 .. R-1
                            if (q < R) {
                                const unsigned c = S.samp[q * ns / R];
                                const bool dup = (q >= 2 && S.samp[(q - 1) * ns / R] == c) ||
                                                 (q + 1 < R && S.samp[(q + 1) * ns / R] == c);
                                bnd[2 * h] = c;
                                bnd[2 * h + 1] = (dup && c != 0xFFFFFFFFu) ? c + 1 : 0u;
                            }
                        }
                        if (lane == 31) bnd[7] = T + 1;  // position 255: no splitter lands there (R <= 128)
                        // Sorted below by the whole CTA, in rank 0's own sample
                        // array (merged into samp above, read by no other CTA).
        #pragma unroll
                        for (int jj = 0; jj < 8; ++jj) S.mysamp[jj * 32 + lane] = bnd[jj];
                    }
                    block_sort_smem_desc(S.mysamp, 256);  // rolled, like the sample sort
                    __syncthreads();
                    if (w == 0) {
                        // The distinct nonzero bounds, in descending order.
                        unsigned nr = 0;
        #pragma unroll 1
                        for (int jj = 0; jj < 8; ++jj) {
                            const unsigned p = jj * 32 + lane;
                            const unsigned v = S.mysamp[p];
                            const bool keep = v != 0u && (p == 0 || v != S.mysamp[p - 1]);
                            const unsigned b = __ballot_sync(kFullMask, keep);
                            if (keep) S.lb[nr + __popc(b & lanemask_lt())] = v;
                            nr += __popc(b);
                        }
                        if (lane == 0) S.nranges = nr;
                    }
                } else if (tid == 0) {
                    S.nranges = 0u;
                }
            }
            cluster_barrier();  // rank 0's range table is out

            if (rank != 0 && tid <= (unsigned)kMaxRanges) {
                if (tid < (unsigned)kMaxRanges)
                    S.lb[tid] = ld_cluster(&S.lb[tid], 0);
                else
                    S.nranges = ld_cluster(&S.nranges, 0);
            }
        }
        if (tid < (unsigned)kMaxRanges) S.rcnt[tid] = 0u;
        __syncthreads();
        nr = S.nranges;
        if (nr) {
            for (unsigned m = lane; m < cw; m += 32) atomicAdd(&S.rcnt[range_of(S.lb, nr, S.keys[w0 + m])], 1u);
        }
        __syncthreads();
        cluster_barrier();  // every CTA's range counts are out

        // part[r][q]: CTA r's keys in range q.  Range q starts at the keys of
        // all lower ranges; this CTA's keys in it follow those of lower ranks.
    #pragma unroll
        for (int h = 0; h < 2; ++h) {
            const unsigned e = tid + h * kClThreads, r = e / kMaxRanges, q = e % kMaxRanges;
            S.part[r][q] = q < nr ? ld_cluster(&S.rcnt[q], r) : 0u;
        }
        __syncthreads();
        if (w == 0) {
            unsigned c[8], tot = 0;
    #pragma unroll
            for (int h = 0; h < 8; ++h) {
                const unsigned q = lane * 8 + h;
                c[h] = 0;
    #pragma unroll
                for (int r = 0; r < kClCtas; ++r) c[h] += S.part[r][q];
                tot += c[h];
            }
            unsigned x = tot;
    #pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(kFullMask, x, o);
                if ((int)lane >= o) x += y;
            }
            unsigned acc = x - tot;
    #pragma unroll
            for (int h = 0; h < 8; ++h) {
                S.rstart[lane * 8 + h] = acc;
                acc += c[h];
            }
            if (lane == 31) S.rstart[kMaxRanges] = acc;
        }
        __syncthreads();
        if (tid < (unsigned)kMaxRanges) {
            unsigned below = 0;
            for (unsigned r = 0; r < rank; ++r) below += S.part[r][tid];
            S.rpos[tid] = S.rstart[tid] + below;
        }
        __syncthreads();
        if (nr) {
            for (unsigned m = lane; m < cw; m += 32) {
                const unsigned u = S.keys[w0 + m];
                out[atomicAdd(&S.rpos[range_of(S.lb, nr, u)], 1u)] = ordered<KIND>(value_of(u));
            }
        }
    }
    // Copies of the k-th key after the keys above it.
    for (unsigned i = total + rank * kClThreads + tid; i < (unsigned)k; i += kClCtas * kClThreads)
        out[i] = ordered<KIND>(value_of(T));
    // The range table for the sort kernel.
    if (rank == 0) {
        RadixPlan* plan = reinterpret_cast<RadixPlan*>(scratch + kRadixCandOffset);
        for (unsigned i = tid; i <= (unsigned)kMaxRanges; i += kClThreads) {
            if (i < nr) plan->lb[i] = S.lb[i];
            if (nr && i <= nr) plan->rstart[i] = S.rstart[i];
        }
        if (tid == 0) plan->nranges = nr;
    }
    cluster_barrier();  // no CTA exits while another may read its shared memory
    if (mode == kClFinal && rank == 0 && tid < (unsigned)kCtrlWords) reinterpret_cast<unsigned*>(rv.ctrl)[tid] = 0u;
}

// Sort kernel: warp w of CTA b sorts range q = b * kSortWarps + w of the
// plan in place, in registers (up to kSortRegCap keys); a range of one value
// is already in order.  A larger range (the sample missed a dense value
// range) is sorted by its CTA in shared memory.
template <int N, int KIND>
__device__ __forceinline__ void warp_sort_range(int32_t* __restrict__ a, unsigned sz, int lane) {
    unsigned v[N];
#pragma unroll
    for (int jj = 0; jj < N; ++jj) {
        const unsigned p = jj * 32 + lane;
        v[jj] = p < sz ? key_of(ordered<KIND>(__ldcg(a + p))) : 0u;
    }
    warp_sort_desc(v, lane);
#pragma unroll
    for (int jj = 0; jj < N; ++jj) {
        const unsigned p = jj * 32 + lane;
        if (p < sz) a[p] = ordered<KIND>(value_of(v[jj]));
    }
}

__device__ __forceinline__ bool single_value_range(const RadixPlan* plan, unsigned q) {
    const unsigned lbq = __ldcg(&plan->lb[q]);
    return q ? __ldcg(&plan->lb[q - 1]) == lbq + 1 : lbq == 0xFFFFFFFFu;
}

template <int KIND>
__global__ void __launch_bounds__(kSortWarps * 32, 1)
radix_sort_kernel(int32_t* __restrict__ out, const unsigned char* __restrict__ scratch, int release) {
    extern __shared__ __align__(16) unsigned radix_sort_smem[];
    grid_dependency_wait();  // launched early (launch_pdl): wait for the previous kernel's writes
    // The plan's last kernel lets the next launch start early only when the
    // caller keeps track of what this one writes.
    if (release) launch_dependents();
    const RadixPlan* plan = reinterpret_cast<const RadixPlan*>(scratch + kRadixCandOffset);
    const unsigned nr = __ldcg(&plan->nranges);
    const unsigned q0 = blockIdx.x * kSortWarps;
    if (q0 >= nr) return;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned q = q0 + w;
    if (q < nr && !single_value_range(plan, q)) {
        const unsigned s0 = __ldcg(&plan->rstart[q]), sz = __ldcg(&plan->rstart[q + 1]) - s0;
        if (sz >= 2 && sz <= 256)
            warp_sort_range<8, KIND>(out + s0, sz, lane);
        else if (sz > 256 && sz <= (unsigned)kSortRegCap)
            warp_sort_range<16, KIND>(out + s0, sz, lane);

    }
    for (unsigned qq = q0; qq < q0 + kSortWarps && qq < nr; ++qq) {
        const unsigned s0 = __ldcg(&plan->rstart[qq]), sz = __ldcg(&plan->rstart[qq + 1]) - s0;
        if (sz <= (unsigned)kSortRegCap || single_value_range(plan, qq)) continue;
        __syncthreads();
        const int L = next_pow2((int)sz);
        for (int i = threadIdx.x; i < L; i += blockDim.x)
            radix_sort_smem[i] = (unsigned)i < sz ? key_of(ordered<KIND>(__ldcg(out + s0 + i))) : 0u;
        block_sort_smem_desc(radix_sort_smem, L);
        for (unsigned i = threadIdx.x; i < sz; i += blockDim.x) out[s0 + i] = ordered<KIND>(value_of(radix_sort_smem[i]));
    }
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
        // The grid of the grid passes: what the SMs hold at once of every
        // one of them (the exact passes' blocks wait on one another).
        const void* passes[] = {reinterpret_cast<const void*>(&radix_filter_kernel<kKeyI32>),
                                reinterpret_cast<const void*>(&radix_filter_kernel<kKeyU32>),
                                reinterpret_cast<const void*>(&radix_filter_kernel<kKeyF32>),
                                reinterpret_cast<const void*>(&radix_exact_kernel<kKeyI32>),
                                reinterpret_cast<const void*>(&radix_exact_kernel<kKeyU32>),
                                reinterpret_cast<const void*>(&radix_exact_kernel<kKeyF32>)};
        int per_sm = 1 << 30;
        for (const void* f : passes) {
            int b = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, f, kRThreads, 0);
            if (e != cudaSuccess) return e;
            if (b < per_sm) per_sm = b;
        }
        const void* cl[] = {reinterpret_cast<const void*>(&radix_cluster_kernel<kKeyI32>),
                            reinterpret_cast<const void*>(&radix_cluster_kernel<kKeyU32>),
                            reinterpret_cast<const void*>(&radix_cluster_kernel<kKeyF32>)};
        const void* so[] = {reinterpret_cast<const void*>(&radix_sort_kernel<kKeyI32>),
                            reinterpret_cast<const void*>(&radix_sort_kernel<kKeyU32>),
                            reinterpret_cast<const void*>(&radix_sort_kernel<kKeyF32>)};
        for (int i = 0; i < 3; ++i) {
            e = cudaFuncSetAttribute(cl[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(ClSmem));
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(so[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(kSortCap * sizeof(unsigned)));
            if (e != cudaSuccess) return e;
        }
        cache[device].grid = sms * (per_sm < 1 ? 1 : per_sm);
    }
    *out = cache[device];
    return cudaSuccess;
}

// Big k: the sorted complemented keys back to the kind's words, in order.
template <int KIND>
__global__ void __launch_bounds__(256) radix_bigk_out_kernel(const uint32_t* __restrict__ sorted, int k,
                                                             int32_t* __restrict__ out) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < k; i += gridDim.x * blockDim.x)
        out[i] = ordered<KIND>(value_of(~__ldg(sorted + i)));
}

template <int KIND>
cudaError_t radix_launch_kind(cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out, void* scratch,
                              size_t cap, int* launches, bool release, uint32_t* bigk) {
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
    constexpr int sort_grid = kMaxRanges / kSortWarps;
    // Every kernel of the plan waits for its predecessor's writes before it
    // reads anything, so each is launched early (launch_pdl), whatever
    // precedes it on the stream.
    if (n <= cap) {
        e = launch_pdl(radix_cluster_kernel<KIND>, kClCtas, kClThreads, cl_smem, s, in, n, k, 0u, out, sc, ucap, kClFull,
                       bigk);
        *launches = 1;
        if (e == cudaSuccess && !bigk) {
            e = launch_pdl(radix_sort_kernel<KIND>, sort_grid, kSortWarps * 32, sort_smem, s, out, sc, release ? 1 : 0);
            *launches = 2;
        }
        return e;
    }
    // Sample rank: k's expected share of the sample, lam, plus four
    // standard deviations plus 2, so that at least k keys are >= t unless
    // the sample holds j or more of the input's k largest (a Poisson(lam)
    // tail: about 6e-5 at lam = 0.66, k = 1000 of 1e8; the exact passes
    // then take over).  The filter keeps about j * n / kSampleKeys keys, so
    // a small k's final usually fits one CTA.
    const double lam = (double)k * (double)kSampleKeys / (double)n;
    const double jd = std::ceil(lam + 4.0 * std::sqrt(lam) + 2.0);
    unsigned j = jd >= (double)kSampleKeys ? kSampleKeys : (unsigned)jd;
    const int opt_j = radix_sample_rank_option();
    if (opt_j > 0) j = (unsigned)opt_j < kSampleKeys ? (unsigned)opt_j : kSampleKeys;
    const size_t per_block = (size_t)kRThreads * kRU * 4;
    size_t grid = (n + per_block - 1) / per_block;
    if (grid > (size_t)f.grid) grid = f.grid;
    if (grid < 1) grid = 1;
    const unsigned g = (unsigned)grid;
    e = launch_pdl(radix_cluster_kernel<KIND>, kClCtas, kClThreads, cl_smem, s, in, n, k, j, out, sc, ucap, kClSample,
                   (uint32_t*)nullptr);
    if (e == cudaSuccess) e = launch_pdl(radix_filter_kernel<KIND>, g, kRThreads, 0, s, in, n, k, sc, ucap);
    if (e == cudaSuccess) e = launch_pdl(radix_exact_kernel<KIND>, g, kRThreads, 0, s, in, n, k, sc, ucap);
    if (e == cudaSuccess)
        e = launch_pdl(radix_cluster_kernel<KIND>, kClCtas, kClThreads, cl_smem, s, in, n, k, 0u, out, sc, ucap, kClFinal,
                       bigk);
    *launches = 4;
    if (e == cudaSuccess && !bigk) {
        e = launch_pdl(radix_sort_kernel<KIND>, sort_grid, kSortWarps * 32, sort_smem, s, out, sc, release ? 1 : 0);
        *launches = 5;
    }
    return e;
}

}  // namespace

cudaError_t radix_launch(cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out, void* scratch,
                         size_t cap, int* launches, bool release, int kind, uint32_t* bigk) {
    if (kind == kKeyU32) return radix_launch_kind<kKeyU32>(s, in, n, k, out, scratch, cap, launches, release, bigk);
    if (kind == kKeyF32) return radix_launch_kind<kKeyF32>(s, in, n, k, out, scratch, cap, launches, release, bigk);
    return radix_launch_kind<kKeyI32>(s, in, n, k, out, scratch, cap, launches, release, bigk);
}

cudaError_t radix_bigk_out(cudaStream_t s, const uint32_t* sorted, int k, int32_t* out, int kind) {
    const int grid = (k + 255) / 256 < 1024 ? (k + 255) / 256 : 1024;
    if (kind == kKeyU32) radix_bigk_out_kernel<kKeyU32><<<grid, 256, 0, s>>>(sorted, k, out);
    else if (kind == kKeyF32) radix_bigk_out_kernel<kKeyF32><<<grid, 256, 0, s>>>(sorted, k, out);
    else radix_bigk_out_kernel<kKeyI32><<<grid, 256, 0, s>>>(sorted, k, out);
    return cudaGetLastError();
}

}  // namespace topk
