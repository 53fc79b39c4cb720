// Two-stage reductions -- sum, max, min -- over int32 and float32, in one
// launch ("CUDA reduction, complete guide": the warp-shuffle level and the
// multi-level reduction system; "CUDA parallel optimisation: TopK",
// section 6: the two-stage pattern reused for other statistics).
//
// Stage 1: a persistent grid; every thread streams its 16-byte vectors of
// the aligned body (8 loads in flight) into a private accumulator; warp
// shuffles and then shared memory combine a block, which writes its partial.
// Stage 2: the last block to finish (atomic ticket) combines the partials
// and writes the result.  No block waits for another.
//
// Results:
//   int32 sum   exact, in int64 (no wrap).
//   int32 max/min.
//   float32 sum each vector's four values added pairwise, the vector sums
//               added with compensation (Neumaier) over each thread's
//               batches of 32 elements, folded into a double per thread,
//               then combined in double.  Error <= 2^-22 sum|x| plus the
//               double rounding of the folds; +-inf and NaN propagate as in
//               IEEE arithmetic (inf + -inf = NaN).  A batch whose float
//               partial sum would pass FLT_MAX (values near 1e37 and more)
//               overflows to inf.
//   float32 max/min  IEEE 754-2019 maximum/minimum: any NaN gives NaN (the
//               canonical quiet NaN); -0 is below +0.  Exact.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "topk_device.cuh"
#include "topk_internal.h"

namespace topk {

namespace {

constexpr int kThreads = 512;
constexpr int kRU = 8;  // 16-byte loads in flight per thread

// ---- accumulator policies ----

// Exact int32 sum without 64-bit arithmetic per element: x = hi * 2^16 + lo
// with hi = x >> 16 (arithmetic) and lo = x & 0xFFFF; a batch of 32
// elements keeps |sum hi| < 2^20 and sum lo < 2^21 in 32-bit registers, and
// end_batch folds them into the int64 total.
struct SumI32 {
    struct Acc {
        long long total;
        unsigned lo;
        int hi;
    };
    __device__ static Acc identity() { return Acc{0, 0u, 0}; }
    __device__ static void add1(Acc& a, int x, bool ok) {
        if (ok) {
            a.lo += (unsigned)x & 0xFFFFu;
            a.hi += x >> 16;
        }
    }
    __device__ static void add(Acc& a, const int4& v, bool ok) {
        add1(a, v.x, ok);
        add1(a, v.y, ok);
        add1(a, v.z, ok);
        add1(a, v.w, ok);
    }
    __device__ static void end_batch(Acc& a) {
        a.total += (long long)a.hi * 65536 + (long long)a.lo;
        a.lo = 0u;
        a.hi = 0;
    }
    __device__ static Acc combine(Acc a, Acc b) { return Acc{a.total + b.total, 0u, 0}; }
    __device__ static Acc shfl_down(Acc a, int o) { return Acc{__shfl_down_sync(kFullMask, a.total, o), 0u, 0}; }
};

template <bool Max>
struct ExtI32 {
    using Acc = int;
    __device__ static Acc identity() { return Max ? INT_MIN : INT_MAX; }
    __device__ static int pick(int a, int b) { return Max ? kmax(a, b) : kmin(a, b); }
    __device__ static void add(Acc& a, const int4& v, bool ok) {
        if (ok) a = pick(a, pick(pick(v.x, v.y), pick(v.z, v.w)));
    }
    __device__ static void add1(Acc& a, int x, bool ok) {
        if (ok) a = pick(a, x);
    }
    __device__ static void end_batch(Acc&) {}
    __device__ static Acc combine(Acc a, Acc b) { return pick(a, b); }
    __device__ static Acc shfl_down(Acc a, int o) { return __shfl_down_sync(kFullMask, a, o); }
};

// Float sum: each vector's four values are added pairwise in float32, and
// the vector sum goes into (s, c), the running compensated (Neumaier) sum of
// the batch; d is the thread's double total.  A vector whose sum is not
// finite is classified element by element: `special` collects +inf (1),
// -inf (2) and NaN (4) inputs, and its finite elements are added one by one.
struct SumF32 {
    struct Acc {
        float s, c;
        double d;
        unsigned special;
    };
    __device__ static Acc identity() { return Acc{0.0f, 0.0f, 0.0, 0u}; }
    __device__ static void neumaier(Acc& a, float x) {
        const float t = a.s + x;
        a.c += fabsf(a.s) >= fabsf(x) ? (a.s - t) + x : (x - t) + a.s;
        a.s = t;
    }
    __device__ static void add1f(Acc& a, float x, bool ok) {
        if (!ok) return;
        if (!isfinite(x)) {
            a.special |= isnan(x) ? 4u : (x > 0.0f ? 1u : 2u);
            return;
        }
        neumaier(a, x);
    }
    __device__ static void add(Acc& a, const int4& v, bool ok) {
        if (!ok) return;
        const float x = __int_as_float(v.x), y = __int_as_float(v.y), z = __int_as_float(v.z),
                    w = __int_as_float(v.w);
        const float sum = (x + y) + (z + w);
        if (isfinite(sum)) {
            neumaier(a, sum);
        } else {
            add1f(a, x, true);
            add1f(a, y, true);
            add1f(a, z, true);
            add1f(a, w, true);
        }
    }
    __device__ static void add1(Acc& a, int x, bool ok) { add1f(a, __int_as_float(x), ok); }
    __device__ static void end_batch(Acc& a) {
        a.d += (double)a.s + (double)a.c;
        a.s = 0.0f;
        a.c = 0.0f;
    }
    __device__ static Acc combine(Acc a, Acc b) { return Acc{0.0f, 0.0f, a.d + b.d, a.special | b.special}; }
    __device__ static Acc shfl_down(Acc a, int o) {
        return Acc{0.0f, 0.0f, __shfl_down_sync(kFullMask, a.d, o), __shfl_down_sync(kFullMask, a.special, o)};
    }
};

// Float max/min on signed-integer keys: negative floats get their magnitude
// bits flipped, so integer order is float order with -0 below +0, positive
// NaNs above +inf and negative NaNs below -inf.  Tracking both the largest
// and the smallest key therefore also tells whether any NaN was seen.
__device__ __forceinline__ int ikey(int b) { return b ^ ((b >> 31) & 0x7FFFFFFF); }
constexpr int kKeyPosInf = 0x7F800000;
constexpr int kKeyNegInf = (int)(0xFF800000u ^ 0x7FFFFFFFu);
template <bool Max>
struct ExtF32 {
    struct Acc {
        int hi, lo;
    };
    __device__ static Acc identity() { return Acc{INT_MIN, INT_MAX}; }
    __device__ static void add1(Acc& a, int b, bool ok) {
        if (!ok) return;
        const int k = ikey(b);
        a.hi = kmax(a.hi, k);
        a.lo = kmin(a.lo, k);
    }
    __device__ static void add(Acc& a, const int4& v, bool ok) {
        if (!ok) return;
        const int k0 = ikey(v.x), k1 = ikey(v.y), k2 = ikey(v.z), k3 = ikey(v.w);
        a.hi = kmax(a.hi, kmax(kmax(k0, k1), kmax(k2, k3)));
        a.lo = kmin(a.lo, kmin(kmin(k0, k1), kmin(k2, k3)));
    }
    __device__ static void end_batch(Acc&) {}
    __device__ static Acc combine(Acc a, Acc b) { return Acc{kmax(a.hi, b.hi), kmin(a.lo, b.lo)}; }
    __device__ static Acc shfl_down(Acc a, int o) {
        return Acc{__shfl_down_sync(kFullMask, a.hi, o), __shfl_down_sync(kFullMask, a.lo, o)};
    }
};

// ---- results ----

__device__ __forceinline__ void finish(const SumI32::Acc& a, void* out) { *static_cast<long long*>(out) = a.total; }
__device__ __forceinline__ void finish(const SumF32::Acc& a, void* out) {
    double r = a.d;
    if ((a.special & 4u) || (a.special & 3u) == 3u)
        r = __longlong_as_double(0x7FF8000000000000ll);
    else if (a.special & 1u)
        r = __longlong_as_double(0x7FF0000000000000ll);
    else if (a.special & 2u)
        r = __longlong_as_double((long long)0xFFF0000000000000ull);
    *static_cast<double*>(out) = r;
}
template <bool Max>
__device__ __forceinline__ void finish_ext_f32(const typename ExtF32<Max>::Acc& a, void* out) {
    double r;
    if (a.hi > kKeyPosInf || a.lo < kKeyNegInf) {
        r = __longlong_as_double(0x7FF8000000000000ll);
    } else {
        const int k = Max ? a.hi : a.lo;
        r = (double)__int_as_float(ikey(k));  // the key map is its own inverse
    }
    *static_cast<double*>(out) = r;
}

template <class Op>
struct Finisher {
    __device__ static void run(const typename Op::Acc& a, void* out) { finish(a, out); }
};
template <bool Max>
struct Finisher<ExtI32<Max>> {
    __device__ static void run(const int& a, void* out) { *static_cast<long long*>(out) = a; }
};
template <bool Max>
struct Finisher<ExtF32<Max>> {
    __device__ static void run(const typename ExtF32<Max>::Acc& a, void* out) { finish_ext_f32<Max>(a, out); }
};

// ---- the kernel ----

// Scratch: the ticket lives in the control line (zero between launches; the
// last block resets it), the block partials after the control area.
constexpr size_t kTicketOffset = kI32CtrlOffset + 64;
constexpr size_t kPartialOffset = kI32CandOffset;
constexpr int kSlotBytes = 32;

template <class Op>
__device__ __forceinline__ typename Op::Acc warp_combine(typename Op::Acc a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = Op::combine(a, Op::shfl_down(a, o));
    return a;
}

template <class Op>
__global__ void __launch_bounds__(kThreads, 2)
reduce_kernel(const int32_t* __restrict__ in, size_t n, void* __restrict__ out, unsigned char* __restrict__ scratch) {
    using Acc = typename Op::Acc;
    static_assert(sizeof(Acc) <= kSlotBytes, "partial slot");
    __shared__ Acc s_warp[kThreads / 32];
    __shared__ int s_last;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;

    Acc a = Op::identity();
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
        for (int u = 0; u < kRU; ++u) Op::add(a, r[u], base + (size_t)u * blockDim.x + threadIdx.x < nvec);
        Op::end_batch(a);
    }
    if (blockIdx.x == 0 && threadIdx.x < 32) {
        const size_t ns = head + (n - tail0);  // < 8 scalars outside the body
        const size_t pos = (size_t)lane < head ? (size_t)lane : tail0 + (lane - head);
        Op::add1(a, (size_t)lane < ns ? in[pos] : 0, (size_t)lane < ns);
        Op::end_batch(a);
    }

    a = warp_combine<Op>(a);
    if (lane == 0) s_warp[w] = a;
    __syncthreads();
    auto* partials = reinterpret_cast<Acc*>(scratch + kPartialOffset);
    unsigned* ticket = reinterpret_cast<unsigned*>(scratch + kTicketOffset);
    if (w == 0) {
        Acc b = lane < kThreads / 32 ? s_warp[lane] : Op::identity();
        b = warp_combine<Op>(b);
        if (lane == 0) partials[blockIdx.x] = b;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // Stage 2: the last block combines every block's partial.
    Acc c = Op::identity();
    for (unsigned i = threadIdx.x; i < gridDim.x; i += blockDim.x) {
        Acc p;
        const unsigned* src = reinterpret_cast<const unsigned*>(&partials[i]);
        unsigned* dst = reinterpret_cast<unsigned*>(&p);
#pragma unroll
        for (int q = 0; q < (int)(sizeof(Acc) / 4); ++q) dst[q] = __ldcg(src + q);
        c = Op::combine(c, p);
    }
    c = warp_combine<Op>(c);
    __syncthreads();
    if (lane == 0) s_warp[w] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        Acc t = s_warp[0];
        for (int i = 1; i < kThreads / 32; ++i) t = Op::combine(t, s_warp[i]);
        Finisher<Op>::run(t, out);
        *ticket = 0u;
    }
}

template <class Op>
int reduce_grid(int device) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static int cache[kMaxDev];
    if (device < 0 || device >= kMaxDev) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[device] == 0) {
        int sms = 0, b = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, reinterpret_cast<const void*>(&reduce_kernel<Op>),
                                                          kThreads, 0) != cudaSuccess)
            return 0;
        int g = sms * (b < 1 ? 1 : b);
        cache[device] = g > kI32MaxGrid ? kI32MaxGrid : g;
    }
    return cache[device];
}

template <class Op>
cudaError_t launch_reduce(cudaStream_t s, const int32_t* in, size_t n, void* out, void* scratch) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    const int gmax = reduce_grid<Op>(device);
    if (gmax == 0) return cudaErrorUnknown;
    const size_t per_block = (size_t)kThreads * kRU * 4;
    size_t grid = (n + per_block - 1) / per_block;
    if (grid > (size_t)gmax) grid = gmax;
    if (grid < 1) grid = 1;
    reduce_kernel<Op><<<(int)grid, kThreads, 0, s>>>(in, n, out, static_cast<unsigned char*>(scratch));
    return cudaGetLastError();
}

}  // namespace

cudaError_t reduce_launch(cudaStream_t s, const void* in, size_t n, bool is_float, int op, void* out, void* scratch) {
    const auto* p = static_cast<const int32_t*>(in);
    if (!is_float) {
        if (op == 0) return launch_reduce<SumI32>(s, p, n, out, scratch);
        if (op == 1) return launch_reduce<ExtI32<true>>(s, p, n, out, scratch);
        return launch_reduce<ExtI32<false>>(s, p, n, out, scratch);
    }
    if (op == 0) return launch_reduce<SumF32>(s, p, n, out, scratch);
    if (op == 1) return launch_reduce<ExtF32<true>>(s, p, n, out, scratch);
    return launch_reduce<ExtF32<false>>(s, p, n, out, scratch);
}

}  // namespace topk
