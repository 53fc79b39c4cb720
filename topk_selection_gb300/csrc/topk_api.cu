// C ABI of libtopk.so: argument checks, workspace, host-buffer staging and
// dispatch to the kernels.  The contract of every entry point is in
// include/topk.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/topk.h"
#include "topk_internal.h"

static_assert(TOPK_MAX_K == topk::kBigKMax, "the header states the big-k form's limit");

namespace {

std::atomic<unsigned long long> g_launches{0};
std::atomic<int> g_stage2_cap{0};
std::atomic<int> g_radix_cap{0};
std::atomic<int> g_radix_sample_rank{0};
std::atomic<int> g_stream_static{0};
std::atomic<int> g_no_early{0};
std::atomic<int> g_sort_spins{0};
std::atomic<int> g_sort_withhold{0};
std::atomic<int> g_fault_alloc{-1};  // -1: not read yet from TOPK_FAULT_ALLOC

// Fault injection on the host: when set (environment TOPK_FAULT_ALLOC=1 at
// the first allocation, or TOPK_OPT_FAULT_ALLOC), every workspace or staging
// allocation fails as if the device were out of memory.
bool fault_alloc() {
    int v = g_fault_alloc.load(std::memory_order_relaxed);
    if (v < 0) {
        const char* env = std::getenv("TOPK_FAULT_ALLOC");
        v = (env && env[0] == '1') ? 1 : 0;
        int expected = -1;
        g_fault_alloc.compare_exchange_strong(expected, v);
        v = g_fault_alloc.load(std::memory_order_relaxed);
    }
    return v == 1;
}
thread_local int t_last_cuda_error = 0;
thread_local int t_last_early = 0;  // whether this thread's last TopK launch started early

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return TOPK_ERR_CUDA;
}

// Cached device memory for one (device, stream) pair.
struct Workspace {
    void* ctrl_cand = nullptr;  // int32 TopK scratch: control words, block maxima, candidates
    size_t ctrl_cand_bytes = 0;
    void* stage_in = nullptr;   // device copy of a host input
    size_t stage_in_bytes = 0;
    void* stage_out = nullptr;  // device buffer for host outputs
    size_t stage_out_bytes = 0;
    void* items = nullptr;      // topk_items_f32 scratch
    size_t items_bytes = 0;
    // What the last launch on this stream writes, when that launch lets its
    // successor start early (up to two ranges): a successor that starts early
    // must not read it.  After any other launch of this library on the
    // stream, and before the first one, the record covers all memory, so
    // that the next launch does not start early.
    const void* stream_out[2] = {nullptr, nullptr};
    size_t stream_out_bytes[2] = {SIZE_MAX, 0};
    void* bigk = nullptr;       // large-k TopK beyond the range plan: two k-word buffers
    size_t bigk_bytes = 0;
    void* sort = nullptr;       // topk_sort_u32 scratch (its header zero between calls)
    size_t sort_bytes = 0;
    unsigned sort_epoch = 0;    // tags the sort's look-back words, one per call
};

std::mutex g_ws_mutex;
std::map<std::pair<int, uintptr_t>, Workspace> g_ws;

int grow(void** p, size_t* have, size_t need) {
    if (*have >= need) return TOPK_OK;
    if (fault_alloc()) {
        t_last_cuda_error = (int)cudaErrorMemoryAllocation;
        return TOPK_ERR_NO_MEMORY;
    }
    if (*p) {
        cudaError_t e = cudaFree(*p);
        *p = nullptr;
        *have = 0;
        if (e != cudaSuccess) return cuda_fail(e);
    }
    cudaError_t e = cudaMalloc(p, need);
    if (e != cudaSuccess) {
        *p = nullptr;
        cudaGetLastError();
        t_last_cuda_error = (int)e;
        return TOPK_ERR_NO_MEMORY;
    }
    *have = need;
    return TOPK_OK;
}

// Workspace for (current device, stream); sizes grow monotonically.
int workspace(cudaStream_t s, int device, size_t ctrl_cand, size_t in_bytes, size_t out_bytes, Workspace** out) {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    Workspace& w = g_ws[{device, reinterpret_cast<uintptr_t>(s)}];
    if (ctrl_cand && w.ctrl_cand_bytes < ctrl_cand) {
        int rc = grow(&w.ctrl_cand, &w.ctrl_cand_bytes, ctrl_cand);
        if (rc != TOPK_OK) return rc;
        // The control words and block-maximum slots must start at zero; the
        // kernels leave them so.
        cudaError_t e = cudaMemsetAsync(w.ctrl_cand, 0, topk::kI32ResetEnd, s);  // status word included
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (in_bytes) {
        int rc = grow(&w.stage_in, &w.stage_in_bytes, in_bytes);
        if (rc != TOPK_OK) return rc;
    }
    if (out_bytes) {
        int rc = grow(&w.stage_out, &w.stage_out_bytes, out_bytes);
        if (rc != TOPK_OK) return rc;
    }
    *out = &w;
    return TOPK_OK;
}

// True when p is host memory (pageable or pinned) rather than device or
// managed memory.
int is_host_pointer(const void* p, bool* host) {
    cudaPointerAttributes a;
    std::memset(&a, 0, sizeof(a));
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e == cudaErrorInvalidValue) {  // unregistered host memory on some drivers
        cudaGetLastError();
        *host = true;
        return TOPK_OK;
    }
    if (e != cudaSuccess) return cuda_fail(e);
    *host = a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeUnregistered;
    return TOPK_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Whether a launch reading `in` may start early (see i32_launch): when `in`
// does not overlap what the stream's last releasing launch writes.  Records
// what this launch writes (ranges a and b; b may be empty) for the next one.
// Only launches that release their successors early may call it; host
// inputs are staged by a copy, which never overlaps a kernel.
bool early_start(Workspace* w, const void* in, size_t in_bytes, const void* a, size_t a_bytes, const void* b,
                 size_t b_bytes) {
    t_last_early = 0;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    bool ok = true;
    for (int i = 0; i < 2; ++i) ok = ok && !overlaps(in, in_bytes, w->stream_out[i], w->stream_out_bytes[i]);
    if (g_no_early.load(std::memory_order_relaxed)) ok = false;
    w->stream_out[0] = a;
    w->stream_out_bytes[0] = a_bytes;
    w->stream_out[1] = b;
    w->stream_out_bytes[1] = b_bytes;
    t_last_early = ok ? 1 : 0;
    return ok;
}

// Record that the last launch on w's stream does not release its successor
// early: the next launch there must not start early, whatever it reads.
void mark_not_released(Workspace* w) {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    w->stream_out[0] = nullptr;
    w->stream_out_bytes[0] = SIZE_MAX;
    w->stream_out[1] = nullptr;
    w->stream_out_bytes[1] = 0;
    t_last_early = 0;
}

}  // namespace

namespace topk {
int stage2_cap_option() { return g_stage2_cap.load(std::memory_order_relaxed); }
int radix_cap_option() { return g_radix_cap.load(std::memory_order_relaxed); }
int radix_sample_rank_option() { return g_radix_sample_rank.load(std::memory_order_relaxed); }
int stream_static_option() { return g_stream_static.load(std::memory_order_relaxed); }
int sort_spins_option() { return g_sort_spins.load(std::memory_order_relaxed); }
int sort_withhold_option() { return g_sort_withhold.load(std::memory_order_relaxed); }
void note_cuda_error(int err) { t_last_cuda_error = err; }
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
void note_unreleased_launch(int device, cudaStream_t s) {
    Workspace* w = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_ws_mutex);
        auto it = g_ws.find({device, reinterpret_cast<uintptr_t>(s)});
        if (it == g_ws.end()) {
            // A workspace made later starts with a record that covers all memory.
            t_last_early = 0;
            return;
        }
        w = &it->second;
    }
    mark_not_released(w);
}
}  // namespace topk

extern "C" {

namespace {

// Body of topk_i32, topk_u32 and topk_f32: n 32-bit words in, k words out,
// ordered as `kind` says (KeyKind).
int topk_words(const int32_t* in, size_t n, int k, int32_t* out, struct CUstream_st* stream, int kind) {
    if (!in || !out || n == 0 || k < 1 || (size_t)k > n) return TOPK_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 3u) return TOPK_ERR_INVALID_ARG;
    if (overlaps(in, n * sizeof(int32_t), out, (size_t)k * sizeof(int32_t))) return TOPK_ERR_INVALID_ARG;
    if (k > TOPK_MAX_K) return TOPK_ERR_UNSUPPORTED;
    if (n > (size_t(1) << 40)) return TOPK_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e);
    bool in_host = false, out_host = false;
    int rc = is_host_pointer(in, &in_host);
    if (rc != TOPK_OK) return rc;
    rc = is_host_pointer(out, &out_host);
    if (rc != TOPK_OK) return rc;

    topk::I32Plan plan;
    e = topk::i32_plan(device, n, k <= 128 ? k : 128, &plan, kind);
    if (e != cudaSuccess) return cuda_fail(e);
    // One workspace serves both plans (k <= 128 streams; larger k use radix select).
    size_t ctrl_cand = topk::i32_scratch_bytes(plan.max_grid);
    const size_t radix_bytes = topk::radix_scratch_bytes(topk::kRadixCap);
    if (radix_bytes > ctrl_cand) ctrl_cand = radix_bytes;
    Workspace* w = nullptr;
    rc = workspace(s, device, ctrl_cand, in_host ? n * sizeof(int32_t) : 0,
                   out_host ? (size_t)k * sizeof(int32_t) : 0, &w);
    if (rc != TOPK_OK) return rc;

    const int32_t* din = in;
    int32_t* dout = out;
    if (in_host) {
        e = cudaMemcpyAsync(w->stage_in, in, n * sizeof(int32_t), cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e);
        din = static_cast<const int32_t*>(w->stage_in);
    }
    if (out_host) dout = static_cast<int32_t*>(w->stage_out);

    int launches = 1;
    if (k > topk::kRadixMaxK) {
        // Beyond the range plan's k: the plan leaves the answer's keys
        // unordered in a buffer, the LSD radix sort orders them, and a last
        // kernel writes them out.  None of these releases its successor.
        const size_t need_sort = topk::sort_scratch_bytes((size_t)k, false);
        unsigned epoch = 0;
        {
            std::lock_guard<std::mutex> lock(g_ws_mutex);
            rc = grow(&w->bigk, &w->bigk_bytes, 2 * (size_t)k * sizeof(uint32_t));
            if (rc == TOPK_OK && w->sort_bytes < need_sort) {
                rc = grow(&w->sort, &w->sort_bytes, need_sort);
                if (rc == TOPK_OK) {
                    e = cudaMemsetAsync(w->sort, 0, topk::kSortHeaderBytes, s);
                    if (e != cudaSuccess) return cuda_fail(e);
                }
            }
            epoch = ++w->sort_epoch;
        }
        if (rc != TOPK_OK) return rc;
        mark_not_released(w);
        auto* a = static_cast<uint32_t*>(w->bigk);
        uint32_t* b = a + k;
        auto* status = reinterpret_cast<unsigned*>(static_cast<char*>(w->ctrl_cand) + topk::kI32StatusOffset);
        e = topk::radix_launch(s, din, n, k, dout, w->ctrl_cand, topk::kRadixCap, &launches, false, kind, a);
        int sl = 0;
        if (e == cudaSuccess) e = topk::sort_launch(s, a, nullptr, (size_t)k, b, nullptr, w->sort, epoch, status, &sl);
        if (e == cudaSuccess) e = topk::radix_bigk_out(s, b, k, dout, kind);
        launches += sl + 1;
    } else if (k <= 128) {
        // The streaming kernel may start while the previous one on this stream
        // finishes, reading its input early: not when that input is the
        // previous launch's output (a chain of TopKs).
        const bool early = early_start(w, din, n * sizeof(int32_t), dout, (size_t)k * sizeof(int32_t), nullptr, 0) &&
                           !in_host;
        e = topk::i32_launch(plan, s, din, n, k, dout, w->ctrl_cand, early, true);
    } else {
        // The large-k kernels let their successors start early too (each of
        // them waits before reading anything): a streaming launch after this
        // one must know what it writes.
        early_start(w, din, 0, dout, (size_t)k * sizeof(int32_t), nullptr, 0);
        t_last_early = 0;  // every kernel of the plan waits before it reads its input
        e = topk::radix_launch(s, din, n, k, dout, w->ctrl_cand, topk::kRadixCap, &launches, true, kind);
    }
    g_launches.fetch_add((unsigned long long)launches, std::memory_order_relaxed);
    if (e != cudaSuccess) return cuda_fail(e);

    if (out_host) {
        e = cudaMemcpyAsync(out, dout, (size_t)k * sizeof(int32_t), cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (in_host || out_host) {
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return TOPK_OK;
}

}  // namespace

int topk_i32(const int32_t* in, size_t n, int k, int32_t* out, struct CUstream_st* stream) {
    return topk_words(in, n, k, out, stream, topk::kKeyI32);
}

int topk_u32(const uint32_t* in, size_t n, int k, uint32_t* out, struct CUstream_st* stream) {
    return topk_words(reinterpret_cast<const int32_t*>(in), n, k, reinterpret_cast<int32_t*>(out), stream,
                      topk::kKeyU32);
}

int topk_f32(const float* in, size_t n, int k, float* out, struct CUstream_st* stream) {
    return topk_words(reinterpret_cast<const int32_t*>(in), n, k, reinterpret_cast<int32_t*>(out), stream,
                      topk::kKeyF32);
}

namespace {

// Shared body of topk_reduce_i32 / topk_reduce_f32: in holds n 4-byte
// values, out one 8-byte result.
int reduce_common(const void* in, size_t n, int op, void* out, bool is_float, struct CUstream_st* stream) {
    if (!in || !out || n == 0 || op < TOPK_REDUCE_SUM || op > TOPK_REDUCE_MIN) return TOPK_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(in) & 3u) || (reinterpret_cast<uintptr_t>(out) & 7u)) return TOPK_ERR_INVALID_ARG;
    if (overlaps(in, n * 4, out, 8)) return TOPK_ERR_INVALID_ARG;
    if (n > (size_t(1) << 40)) return TOPK_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e);
    bool in_host = false, out_host = false;
    int rc = is_host_pointer(in, &in_host);
    if (rc == TOPK_OK) rc = is_host_pointer(out, &out_host);
    if (rc != TOPK_OK) return rc;
    Workspace* w = nullptr;
    rc = workspace(s, device, topk::kReduceScratchBytes, in_host ? n * 4 : 0, out_host ? 8 : 0, &w);
    if (rc != TOPK_OK) return rc;
    const void* din = in;
    void* dout = out;
    if (in_host) {
        e = cudaMemcpyAsync(w->stage_in, in, n * 4, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e);
        din = w->stage_in;
    }
    if (out_host) dout = w->stage_out;
    mark_not_released(w);
    e = topk::reduce_launch(s, din, n, is_float, op, dout, w->ctrl_cand);
    if (e != cudaSuccess) return cuda_fail(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (out_host) {
        e = cudaMemcpyAsync(out, dout, 8, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (in_host || out_host) {
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return TOPK_OK;
}

}  // namespace

int topk_reduce_i32(const int32_t* in, size_t n, int op, int64_t* out, struct CUstream_st* stream) {
    return reduce_common(in, n, op, out, false, stream);
}

int topk_reduce_f32(const float* in, size_t n, int op, double* out, struct CUstream_st* stream) {
    return reduce_common(in, n, op, out, true, stream);
}

int topk_sort_u32(const uint32_t* keys, const uint32_t* vals, size_t n, uint32_t* keys_out, uint32_t* vals_out,
                  struct CUstream_st* stream) {
    if (!keys || !keys_out || n == 0 || (!vals) != (!vals_out)) return TOPK_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(keys) | reinterpret_cast<uintptr_t>(keys_out) |
         reinterpret_cast<uintptr_t>(vals) | reinterpret_cast<uintptr_t>(vals_out)) & 3u)
        return TOPK_ERR_INVALID_ARG;
    const size_t b = n * 4;
    if (overlaps(keys, b, keys_out, b) || (vals && (overlaps(vals, b, vals_out, b) || overlaps(keys, b, vals_out, b) ||
                                                     overlaps(vals, b, keys_out, b) || overlaps(keys_out, b, vals_out, b))))
        return TOPK_ERR_INVALID_ARG;
    if (n > (size_t)0xFFFFFFFFu) return TOPK_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e);
    for (const void* p : {(const void*)keys, (const void*)vals, (const void*)keys_out, (const void*)vals_out}) {
        if (!p) continue;
        bool host = false;
        const int rc = is_host_pointer(p, &host);
        if (rc != TOPK_OK) return rc;
        if (host) return TOPK_ERR_INVALID_ARG;  // device memory only
    }
    Workspace* w = nullptr;
    int rc = workspace(s, device, topk::kI32CandOffset, 0, 0, &w);
    if (rc != TOPK_OK) return rc;
    unsigned epoch = 0;
    {
        std::lock_guard<std::mutex> lock(g_ws_mutex);
        const size_t need = topk::sort_scratch_bytes(n, vals != nullptr);
        if (w->sort_bytes < need) {
            rc = grow(&w->sort, &w->sort_bytes, need);
            if (rc != TOPK_OK) return rc;
            e = cudaMemsetAsync(w->sort, 0, topk::kSortHeaderBytes, s);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        epoch = ++w->sort_epoch;
    }
    auto* status = reinterpret_cast<unsigned*>(static_cast<char*>(w->ctrl_cand) + topk::kI32StatusOffset);
    int launches = 0;
    mark_not_released(w);
    e = topk::sort_launch(s, keys, vals, n, keys_out, vals_out, w->sort, epoch, status, &launches);
    g_launches.fetch_add((unsigned long long)launches, std::memory_order_relaxed);
    if (e != cudaSuccess) return cuda_fail(e);
    return TOPK_OK;
}

int topk_items_f32(const float* score, const int64_t* item, const uint8_t* keep, size_t n, int k, float* out_score,
                   int64_t* out_item, int64_t* out_count, struct CUstream_st* stream) {
    if (!score || !out_score || !out_item || n == 0 || k < 1 || (size_t)k > n) return TOPK_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(score) | reinterpret_cast<uintptr_t>(out_score)) & 3u)
        return TOPK_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(item) | reinterpret_cast<uintptr_t>(out_item) |
         reinterpret_cast<uintptr_t>(out_count)) & 7u)
        return TOPK_ERR_INVALID_ARG;
    const size_t ko = (size_t)k;
    if (overlaps(score, n * 4, out_score, ko * 4) || overlaps(score, n * 4, out_item, ko * 8) ||
        overlaps(out_score, ko * 4, out_item, ko * 8) || (item && overlaps(item, n * 8, out_item, ko * 8)))
        return TOPK_ERR_INVALID_ARG;
    if (k > TOPK_MAX_K_ROWS) return TOPK_ERR_UNSUPPORTED;
    if (n > (size_t)INT32_MAX) return TOPK_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e);
    for (const void* p : {(const void*)score, (const void*)item, (const void*)keep, (const void*)out_score,
                          (const void*)out_item, (const void*)out_count}) {
        if (!p) continue;
        bool host = false;
        const int rc = is_host_pointer(p, &host);
        if (rc != TOPK_OK) return rc;
        if (host) return TOPK_ERR_INVALID_ARG;  // device memory only
    }
    Workspace* w = nullptr;
    int rc = workspace(s, device, topk::kI32CandOffset, 0, 0, &w);
    if (rc != TOPK_OK) return rc;
    const size_t need = topk::items_scratch_bytes(
        n, k, keep != nullptr && !topk::items_fused_filter(score, keep, n, k));
    {
        std::lock_guard<std::mutex> lock(g_ws_mutex);
        rc = grow(&w->items, &w->items_bytes, need);
    }
    if (rc != TOPK_OK) return rc;
    auto* status = reinterpret_cast<unsigned*>(static_cast<char*>(w->ctrl_cand) + topk::kI32StatusOffset);
    int launches = 0;
    mark_not_released(w);
    e = topk::items_launch(s, score, item, keep, n, k, out_score, out_item, out_count, w->items, w->items_bytes,
                           status, &launches);
    g_launches.fetch_add((unsigned long long)launches, std::memory_order_relaxed);
    if (e != cudaSuccess) return cuda_fail(e);
    return TOPK_OK;
}

int topk_rows_f32(const float* in, int rows, int cols, int k, float* vals, int32_t* idx,
                  struct CUstream_st* stream) {
    if (!in || !vals || !idx || rows < 1 || cols < 1 || k < 1 || k > cols) return TOPK_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(vals) | reinterpret_cast<uintptr_t>(idx)) &
        3u)
        return TOPK_ERR_INVALID_ARG;
    const size_t nin = (size_t)rows * (size_t)cols * sizeof(float);
    const size_t nout = (size_t)rows * (size_t)k * sizeof(float);
    if (overlaps(in, nin, vals, nout) || overlaps(in, nin, idx, nout) || overlaps(vals, nout, idx, nout))
        return TOPK_ERR_INVALID_ARG;
    if (k > TOPK_MAX_K_ROWS) return TOPK_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e);
    bool in_host = false, vals_host = false, idx_host = false;
    int rc = is_host_pointer(in, &in_host);
    if (rc == TOPK_OK) rc = is_host_pointer(vals, &vals_host);
    if (rc == TOPK_OK) rc = is_host_pointer(idx, &idx_host);
    if (rc != TOPK_OK) return rc;

    Workspace* w = nullptr;
    const size_t out_stage = (vals_host || idx_host) ? 2 * nout : 0;
    // The row kernels use only the workspace's status word.
    rc = workspace(s, device, topk::kI32CandOffset, in_host ? nin : 0, out_stage, &w);
    if (rc != TOPK_OK) return rc;
    auto* status = reinterpret_cast<unsigned*>(static_cast<char*>(w->ctrl_cand) + topk::kI32StatusOffset);

    const float* din = in;
    float* dvals = vals;
    int32_t* didx = idx;
    if (in_host) {
        e = cudaMemcpyAsync(w->stage_in, in, nin, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e);
        din = static_cast<const float*>(w->stage_in);
    }
    if (vals_host) dvals = static_cast<float*>(w->stage_out);
    if (idx_host) didx = reinterpret_cast<int32_t*>(static_cast<char*>(w->stage_out) + nout);

    // The streamed row kernel (k <= 128) starts early and releases its
    // successors like the int32 streaming kernel.
    bool early = false;
    if (k <= 128)
        early = early_start(w, din, nin, dvals, nout, didx, nout) && !in_host;
    else
        mark_not_released(w);
    e = topk::rows_launch(s, din, rows, cols, k, dvals, didx, status, early, k <= 128 ? topk::kRowsRelease : 0);
    if (e != cudaSuccess) return cuda_fail(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);

    if (vals_host) {
        e = cudaMemcpyAsync(vals, dvals, nout, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (idx_host) {
        e = cudaMemcpyAsync(idx, didx, nout, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (in_host || vals_host || idx_host) {
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return TOPK_OK;
}

int topk_check_stream(struct CUstream_st* stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    void* words[2] = {nullptr, nullptr};
    {
        std::lock_guard<std::mutex> lock(g_ws_mutex);
        auto it = g_ws.find({device, reinterpret_cast<uintptr_t>(s)});
        if (it != g_ws.end() && it->second.ctrl_cand)
            words[0] = static_cast<char*>(it->second.ctrl_cand) + topk::kI32StatusOffset;
    }
    if (void* na = topk::noalloc_scratch_if_ready(device)) words[1] = static_cast<char*>(na) + topk::kI32StatusOffset;
    int rc = TOPK_OK;
    for (void* w : words) {
        if (!w) continue;
        unsigned v = 0;
        e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e);
        if (v != 0) {
            rc = TOPK_ERR_DEVICE_TIMEOUT;
            e = cudaMemset(w, 0, sizeof(v));
            if (e != cudaSuccess) return cuda_fail(e);
        }
    }
    return rc;
}

int topk_set_option(int option, int value) {
    switch (option) {
        case TOPK_OPT_STAGE2_CAP:
            if (value != 0 && (value < 2 || (value & (value - 1)) != 0)) return TOPK_ERR_INVALID_ARG;
            g_stage2_cap.store(value, std::memory_order_relaxed);
            return TOPK_OK;
        case TOPK_OPT_RADIX_CAP:
            if (value < 0) return TOPK_ERR_INVALID_ARG;
            g_radix_cap.store(value, std::memory_order_relaxed);
            return TOPK_OK;
        case TOPK_OPT_RADIX_SAMPLE_RANK:
            if (value < 0) return TOPK_ERR_INVALID_ARG;
            g_radix_sample_rank.store(value, std::memory_order_relaxed);
            return TOPK_OK;
        case TOPK_OPT_NO_EARLY_START:
            if (value != 0 && value != 1) return TOPK_ERR_INVALID_ARG;
            g_no_early.store(value, std::memory_order_relaxed);
            return TOPK_OK;
        case TOPK_OPT_SORT_SPINS:
            if (value < 0) return TOPK_ERR_INVALID_ARG;
            g_sort_spins.store(value, std::memory_order_relaxed);
            return TOPK_OK;
        case TOPK_OPT_SORT_WITHHOLD:
            if (value != 0 && value != 1) return TOPK_ERR_INVALID_ARG;
            g_sort_withhold.store(value, std::memory_order_relaxed);
            return TOPK_OK;
        case TOPK_OPT_FAULT_ALLOC:
            if (value != 0 && value != 1) return TOPK_ERR_INVALID_ARG;
            g_fault_alloc.store(value, std::memory_order_relaxed);
            return TOPK_OK;
        case TOPK_OPT_STREAM_STATIC:
            if (value < 0 || value > 101) return TOPK_ERR_INVALID_ARG;
            g_stream_static.store(value, std::memory_order_relaxed);
            return TOPK_OK;
        default:
            return TOPK_ERR_INVALID_ARG;
    }
}

const char* topk_status_string(int status) {
    switch (status) {
        case TOPK_OK: return "ok";
        case TOPK_ERR_INVALID_ARG: return "invalid argument";
        case TOPK_ERR_UNSUPPORTED: return "unsupported size";
        case TOPK_ERR_NO_MEMORY: return "out of device memory";
        case TOPK_ERR_CUDA: return "CUDA error";
        case TOPK_ERR_DEVICE_TIMEOUT: return "a device-side wait gave up";
        default: return "unknown status";
    }
}

int topk_last_cuda_error(void) { return t_last_cuda_error; }

int topk_last_launch_early(void) { return t_last_early; }

int topk_release_workspace(void) {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    int rc = TOPK_OK;
    int prev = -1;
    cudaGetDevice(&prev);
    for (auto& kv : g_ws) {
        Workspace& w = kv.second;
        cudaSetDevice(kv.first.first);
        for (void* p : {w.ctrl_cand, w.stage_in, w.stage_out, w.items, w.sort, w.bigk})
            if (p && cudaFree(p) != cudaSuccess) rc = TOPK_ERR_CUDA;
    }
    g_ws.clear();
    if (prev >= 0) cudaSetDevice(prev);
    return rc;
}

unsigned long long topk_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
