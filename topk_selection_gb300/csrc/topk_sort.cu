// LSD radix sort of uint32 keys, optionally carrying uint32 values
// ("GPU radix sort": 8-bit digits, four passes for 32-bit keys, per-block
// shared-memory histograms; its extensions section adds key-value pairs).
//
// GB300 form: one histogram pass for all four digits, then one launch per
// digit in which every tile of 8192 keys
//   1. takes the next tile id from a counter (so a tile only ever waits for
//      tiles whose blocks are already running),
//   2. ranks its keys stably: per warp, keys go slot by slot (32
//      consecutive keys per slot); each lane ORs its bit into its warp's
//      shared word for its digit, so the word is the mask of lanes with that
//      digit and a key's rank among equal digits follows input order; warps
//      then add the counts of the warps before them,
//   3. publishes its per-digit counts as soon as the warps' counts give
//      them, and places its keys (and values) in shared memory in digit
//      order,
//   4. looks back over earlier tiles for the keys of each digit before it
//      (decoupled look-back: a tile's word says "my count" or "count of
//      every tile up to me"), 16 words per digit per round trip, now that
//      no key is held in registers, and writes its keys out, so that keys of
//      one digit go to consecutive addresses.
// The page's printed scatter increments shared counters without atomics;
// only its plan (digits, passes, histograms) is kept.
//
// Look-back words are 64-bit: status (2 bits), epoch (30 bits: the call and
// pass that wrote it), count (32 bits).  A word from another call or pass
// reads as "not ready", so the array never needs clearing.  Every wait is
// bounded: after kSpins polls the tile records kStatusWaitTimeout in the
// status word and goes on with what it has (the result is then invalid, and
// topk_check_stream reports it).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "topk_device.cuh"
#include "topk_internal.h"

namespace topk {

int sort_withhold_option();  // test option TOPK_OPT_SORT_WITHHOLD (topk_api.cu)

namespace {

constexpr int kST = 512;            // threads per tile
constexpr int kSW = kST / 32;       // warps per tile
constexpr int kSI = 16;             // keys per thread (8192-key tiles: measured best of 256..1024 x 8..24)
constexpr int kTile = kST * kSI;    // keys per tile
constexpr int kRadix = 256;
constexpr int kSpins = 1 << 22;     // polls of one look-back word before giving up
constexpr int kLookW = 16;          // look-back words read per digit per round trip
constexpr int kHT = 512, kHU = 8;   // histogram pass: threads, 16-byte loads in flight
constexpr int kHR = 8;              // histogram pass: copies of each digit histogram

constexpr unsigned long long kAgg = 1ull << 62;   // word holds this tile's count
constexpr unsigned long long kIncl = 2ull << 62;  // word holds the count up to and including this tile

struct SortHeader {
    unsigned hist[4][kRadix];   // digit counts (zero between calls)
    unsigned base[4][kRadix];   // where each digit's keys start, per pass
    unsigned ticket;            // histogram pass blocks done (zero between calls)
    unsigned tile_counter[4];   // next tile id, per pass (zero between calls)
};
static_assert(sizeof(SortHeader) <= kSortHeaderBytes, "sort header");

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ---- pass 0: histograms of all four digits, then the digit bases ----

__global__ void __launch_bounds__(kHT, 2)
sort_hist_kernel(const uint32_t* __restrict__ keys, size_t n, SortHeader* __restrict__ h) {
    // kHR copies of each digit histogram, bin b of copy r at word b * kHR + r
    // with r = lane % kHR: lanes of different copies never share a bank, so a
    // warp's 32 random bins meet fewer bank conflicts than in one copy.
    __shared__ unsigned sh[4][kRadix * kHR];
    __shared__ int s_last;
    for (int i = threadIdx.x; i < 4 * kRadix * kHR; i += blockDim.x) (&sh[0][0])[i] = 0u;
    __syncthreads();
    const unsigned r = threadIdx.x % kHR;
    auto add = [&](uint32_t k) {
        atomicAdd(&sh[0][(k & 0xFFu) * kHR + r], 1u);
        atomicAdd(&sh[1][((k >> 8) & 0xFFu) * kHR + r], 1u);
        atomicAdd(&sh[2][((k >> 16) & 0xFFu) * kHR + r], 1u);
        atomicAdd(&sh[3][(k >> 24) * kHR + r], 1u);
    };
    const uintptr_t addr = reinterpret_cast<uintptr_t>(keys);
    size_t head = ((16u - (unsigned)(addr & 15u)) & 15u) >> 2;
    if (head > n) head = n;
    const uint4* body = reinterpret_cast<const uint4*>(keys + head);
    const size_t nvec = (n - head) >> 2, tail0 = head + nvec * 4;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t b = (size_t)blockIdx.x * blockDim.x * kHU; b < nvec; b += stride * kHU) {
        uint4 r[kHU];
#pragma unroll
        for (int u = 0; u < kHU; ++u) {
            const size_t i = b + (size_t)u * blockDim.x + threadIdx.x;
            r[u] = i < nvec ? __ldg(body + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kHU; ++u)
            if (b + (size_t)u * blockDim.x + threadIdx.x < nvec) {
                add(r[u].x);
                add(r[u].y);
                add(r[u].z);
                add(r[u].w);
            }
    }
    if (blockIdx.x == 0 && threadIdx.x < 32) {
        const size_t ns = head + (n - tail0), lane = threadIdx.x;
        if (lane < ns) add(keys[lane < head ? lane : tail0 + (lane - head)]);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * kRadix; i += blockDim.x) {
        const unsigned* c = &sh[i / kRadix][(i % kRadix) * kHR];
        unsigned v = 0;
#pragma unroll
        for (int q = 0; q < kHR; ++q) v += c[q];
        if (v) atomicAdd(&(&h->hist[0][0])[i], v);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&h->ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // Last block: exclusive scans of the four histograms (one warp each).
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (w < 4) {
        unsigned c[8], t = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            c[j] = __ldcg(&h->hist[w][lane * 8 + j]);
            t += c[j];
        }
        unsigned x = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(kFullMask, x, o);
            if (lane >= o) x += y;
        }
        unsigned acc = x - t;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            h->base[w][lane * 8 + j] = acc;
            acc += c[j];
            h->hist[w][lane * 8 + j] = 0u;
        }
    }
    if (threadIdx.x == 0) h->ticket = 0u;
}

// ---- one digit pass ----

template <bool kVals>
__global__ void __launch_bounds__(kST, 2)
sort_pass_kernel(const uint32_t* __restrict__ kin, const uint32_t* __restrict__ vin, uint32_t* __restrict__ kout,
                 uint32_t* __restrict__ vout, size_t n, int shift, SortHeader* __restrict__ h, int pass,
                 unsigned long long* __restrict__ look, unsigned epoch, unsigned ntiles, unsigned* __restrict__ status,
                 int max_spins, int withhold) {
    extern __shared__ __align__(16) uint32_t sort_smem[];
    uint32_t* s_keys = sort_smem;                       // kTile
    uint32_t* s_vals = sort_smem + kTile;               // kTile (with values)
    __shared__ unsigned s_whist[kSW][kRadix];           // per-warp counts, then the warps' offsets
    __shared__ unsigned s_match[kSW][kRadix];           // per-warp lane masks of one slot's digits (zero between slots)
    __shared__ unsigned s_tcount[kRadix];               // this tile's count per digit
    __shared__ unsigned s_texcl[kRadix];                // where each digit starts in the tile
    __shared__ unsigned s_goff[kRadix];                 // where this tile's keys of each digit go
    __shared__ unsigned s_tile;
    __shared__ unsigned s_scan[kSW];

    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        const unsigned t = atomicAdd(&h->tile_counter[pass], 1u);
        s_tile = t;
        if (t == ntiles - 1) h->tile_counter[pass] = 0u;  // every block has its id: reset for the next call
    }
    for (int i = lane; i < kRadix; i += 32) {
        s_whist[w][i] = 0u;
        s_match[w][i] = 0u;
    }
    __syncthreads();
    const unsigned tile = s_tile;
    const size_t tbase = (size_t)tile * kTile;
    const unsigned tcnt = (unsigned)(n - tbase < (size_t)kTile ? n - tbase : (size_t)kTile);

    // Load: warp w owns tile keys [w*256, w*256 + 256), slot i = keys
    // w*256 + i*32 .. +31 (lane order = input order).
    uint32_t key[kSI];
    unsigned rank[kSI];
#pragma unroll
    for (int i = 0; i < kSI; ++i) {
        const unsigned p = (unsigned)(w * 32 * kSI + i * 32 + lane);
        key[i] = p < tcnt ? kin[tbase + p] : 0xFFFFFFFFu;
    }
    // Stable rank within the warp among keys of the same digit, slot by
    // slot: every lane ORs its bit into its warp's word for its digit, so
    // the word is the mask of lanes with that digit and a key's rank among
    // them follows input order; the highest of them adds the group to the
    // warp's count and clears the word.  (Keys past the end take no part.)
    {
        volatile unsigned* cnt = s_whist[w];
        volatile unsigned* match = s_match[w];
        const unsigned bit = 1u << lane;
#pragma unroll
        for (int i = 0; i < kSI; ++i) {
            const unsigned p = (unsigned)(w * 32 * kSI + i * 32 + lane);
            const bool ok = p < tcnt;
            const unsigned d = (key[i] >> shift) & 0xFFu;
            if (ok) atomicOr((unsigned*)&match[d], bit);
            __syncwarp();
            const unsigned peers = ok ? match[d] : bit;
            const unsigned before = ok ? cnt[d] : 0u;
            __syncwarp();
            if (ok && lane == 31 - __clz(peers)) {
                cnt[d] = before + __popc(peers);
                match[d] = 0u;
            }
            rank[i] = before + __popc(peers & (bit - 1u));
            __syncwarp();
        }
    }
    __syncthreads();
    // Per digit: the counts of the warps before each warp and the tile's
    // count, published at once (so that later tiles see it early); then
    // where each digit starts inside the tile.
    const unsigned long long tag = (unsigned long long)(epoch & 0x3FFFFFFFu) << 32;
    if (threadIdx.x < kRadix) {
        const int d = threadIdx.x;
        unsigned acc = 0;
#pragma unroll
        for (int ww = 0; ww < kSW; ++ww) {
            const unsigned c = s_whist[ww][d];
            s_whist[ww][d] = acc;
            acc += c;
        }
        s_tcount[d] = acc;
        if (tile != 0 || !withhold)  // (a test option makes the first tile withhold its word)
            st_relaxed_u64(look + (size_t)tile * kRadix + d, (tile == 0 ? kIncl : kAgg) | tag | acc);
        unsigned x = acc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(kFullMask, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_scan[w] = x;
        s_texcl[d] = x - acc;  // within the warp; warps added below
    }
    __syncthreads();
    if (threadIdx.x < kRadix) {
        unsigned add = 0;
        for (int ww = 0; ww < w; ++ww) add += s_scan[ww];
        s_texcl[threadIdx.x] += add;
    }
    __syncthreads();
    // Keys to shared memory in digit order (stable), then out.
#pragma unroll
    for (int i = 0; i < kSI; ++i) {
        const unsigned p = (unsigned)(w * 32 * kSI + i * 32 + lane);
        if (p < tcnt) {
            const unsigned d = (key[i] >> shift) & 0xFFu;
            const unsigned slot = s_texcl[d] + s_whist[w][d] + rank[i];
            s_keys[slot] = key[i];
            if (kVals) s_vals[slot] = vin[tbase + p];  // read only now: no registers held through the ranking
        }
    }
    __syncthreads();
    // Look back (one thread per digit), now that no key or rank is held in
    // registers: walk back over the tiles before this one, kLookW words per
    // round trip, adding counts until a word that already covers every tile
    // before it.  A word not yet written is read again (bounded).
    if (threadIdx.x < kRadix) {
        const int d = threadIdx.x;
        unsigned excl = 0;
        if (tile != 0) {
            long long j = (long long)tile - 1;
            int spins = 0;
            bool done = false;
            while (!done && j >= 0) {
                unsigned long long v[kLookW];
#pragma unroll
                for (int q = 0; q < kLookW; ++q)
                    v[q] = j - q >= 0 ? ld_relaxed_u64(look + (size_t)(j - q) * kRadix + d) : 0ull;
#pragma unroll
                for (int q = 0; q < kLookW; ++q) {
                    if (done || j < 0) break;
                    if ((v[q] & 0x3FFFFFFF00000000ull) != tag || (v[q] >> 62) == 0) {
                        if (++spins >= max_spins) {  // give up: go on with what has been summed
                            atomicOr(status, kStatusWaitTimeout);
                            done = true;
                        }
                        break;  // read again from j
                    }
                    excl += (unsigned)v[q];
                    --j;
                    if ((v[q] >> 62) == 2) done = true;
                }
            }
            st_relaxed_u64(look + (size_t)tile * kRadix + d, kIncl | tag | (excl + s_tcount[d]));
        }
        s_goff[d] = __ldcg(&h->base[pass][d]) + excl;
    }
    __syncthreads();
    for (unsigned i = threadIdx.x; i < tcnt; i += kST) {
        const uint32_t k = s_keys[i];
        const unsigned d = (k >> shift) & 0xFFu;
        const size_t dst = (size_t)s_goff[d] + (i - s_texcl[d]);
        kout[dst] = k;
        if (kVals) vout[dst] = s_vals[i];
    }
}

struct SortFit {
    int hist_grid = 0;
};

cudaError_t sort_fit(int device, SortFit* out) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static SortFit cache[kMaxDev];
    if (device < 0 || device >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[device].hist_grid == 0) {
        int sms = 0, b = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, reinterpret_cast<const void*>(&sort_hist_kernel), kHT, 0);
        if (e != cudaSuccess) return e;
        for (const void* f : {reinterpret_cast<const void*>(&sort_pass_kernel<true>),
                              reinterpret_cast<const void*>(&sort_pass_kernel<false>)}) {
            e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * kTile * 4);
            if (e != cudaSuccess) return e;
        }
        cache[device].hist_grid = sms * (b < 1 ? 1 : b);
    }
    *out = cache[device];
    return cudaSuccess;
}

}  // namespace

size_t sort_scratch_bytes(size_t n, bool with_vals) {
    const size_t tiles = (n + kTile - 1) / kTile;
    const size_t look = tiles * kRadix * 8;
    const size_t tmp = (n * 4 + 255) / 256 * 256;
    return kSortHeaderBytes + (look + 255) / 256 * 256 + tmp * (with_vals ? 2 : 1);
}

cudaError_t sort_launch(cudaStream_t s, const uint32_t* keys, const uint32_t* vals, size_t n, uint32_t* keys_out,
                        uint32_t* vals_out, void* scratch, unsigned epoch, unsigned* status, int* launches) {
    *launches = 0;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    SortFit f;
    e = sort_fit(device, &f);
    if (e != cudaSuccess) return e;
    auto* base = static_cast<unsigned char*>(scratch);
    auto* h = reinterpret_cast<SortHeader*>(base);
    const size_t tiles = (n + kTile - 1) / kTile;
    auto* look = reinterpret_cast<unsigned long long*>(base + kSortHeaderBytes);
    const size_t look_bytes = (tiles * kRadix * 8 + 255) / 256 * 256;
    auto* tk = reinterpret_cast<uint32_t*>(base + kSortHeaderBytes + look_bytes);
    const size_t tmp = (n * 4 + 255) / 256 * 256;
    auto* tv = vals ? reinterpret_cast<uint32_t*>(base + kSortHeaderBytes + look_bytes + tmp) : nullptr;

    size_t hgrid = (n + (size_t)kHT * kHU * 4 - 1) / ((size_t)kHT * kHU * 4);
    if (hgrid > (size_t)f.hist_grid) hgrid = f.hist_grid;
    if (hgrid < 1) hgrid = 1;
    sort_hist_kernel<<<(int)hgrid, kHT, 0, s>>>(keys, n, h);
    *launches += 1;
    // pass 0: keys -> tmp, 1: tmp -> out, 2: out -> tmp, 3: tmp -> out
    const uint32_t* ki[4] = {keys, tk, keys_out, tk};
    uint32_t* ko[4] = {tk, keys_out, tk, keys_out};
    const uint32_t* vi[4] = {vals, tv, vals_out, tv};
    uint32_t* vo[4] = {tv, vals_out, tv, vals_out};
    const size_t smem = (size_t)(vals ? 2 : 1) * kTile * 4;
    // Polls of one look-back word before a tile gives up (TOPK_OPT_SORT_SPINS
    // lowers it for tests).  A tile that gives up has summed only some of the
    // tiles before it, so its digit offsets are too small but never below the
    // digit's base: every write stays inside [0, n), the order is wrong, and
    // the status word reports it.
    const int opt_spins = sort_spins_option();
    const int spins = opt_spins > 0 ? opt_spins : kSpins;
    const int withhold = sort_withhold_option();
    for (int p = 0; p < 4; ++p) {
        const unsigned ep = (epoch * 4u + (unsigned)p) & 0x3FFFFFFFu;
        if (vals)
            sort_pass_kernel<true><<<(unsigned)tiles, kST, smem, s>>>(ki[p], vi[p], ko[p], vo[p], n, 8 * p, h, p,
                                                                     look, ep, (unsigned)tiles, status, spins, withhold);
        else
            sort_pass_kernel<false><<<(unsigned)tiles, kST, smem, s>>>(ki[p], nullptr, ko[p], nullptr, n, 8 * p, h,
                                                                      p, look, ep, (unsigned)tiles, status, spins, withhold);
        *launches += 1;
    }
    return cudaGetLastError();
}

}  // namespace topk
