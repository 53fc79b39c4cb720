// topk_i32_noalloc: the int32 TopK for callers that may not allocate.
//
// Some callers cannot call cudaMalloc: the enqueue hook of a framework
// plugin that is forbidden to allocate, a process whose device memory has
// been claimed up front by another allocator's pool, or a latency-bound loop
// that cannot afford the implicit synchronisation of cudaMalloc/cudaFree.
// This entry point runs the same kernel as topk_i32, but its scratch (the
// control words, the block maxima and the per-block candidates) lives in the file-scope
// device array below instead of the library's cudaMalloc'd workspace.
//
// The array is part of the module image: every GPU that loads the library
// holds kNoallocScratchBytes of it until the process exits.  Host code must
// not use the array's name as a device address (on the host it names a
// stand-in); its device address is taken once per device with
// cudaGetSymbolAddress and cached.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/topk.h"
#include "topk_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = TOPK_NOALLOC_SCRATCH_BYTES;
static_assert(kNoallocScratchBytes >= topk::i32_scratch_bytes(1),
              "the scratch must hold the control words, block maxima, counts and one block's candidates");
static_assert(kNoallocScratchBytes >= topk::radix_scratch_bytes(TOPK_NOALLOC_MAX_K),
              "the radix plan's candidate buffer must hold at least the largest k keys");
// The candidate buffer of the radix plan here, in keys (the header quotes it).
constexpr size_t kNoallocRadixCap = (kNoallocScratchBytes - topk::radix_scratch_bytes(0)) / sizeof(unsigned);
static_assert(kNoallocRadixCap == 252800, "topk.h states this capacity");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on `device` (which must be current).
// Done once per device, on the first call there.
int scratch_address(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return TOPK_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[device]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            topk::note_cuda_error((int)e);
            return TOPK_ERR_CUDA;
        }
        g_scratch_ptr[device] = p;
    }
    *out = g_scratch_ptr[device];
    return TOPK_OK;
}

bool is_device_memory(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

}  // namespace

namespace topk {
// Device address of the no-alloc scratch on `device`, or null if no call
// has set it up yet.
void* noalloc_scratch_if_ready(int device) {
    if (device < 0 || device >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    return g_scratch_ptr[device];
}
}  // namespace topk

extern "C" int topk_i32_noalloc(const int32_t* in, size_t n, int k, int32_t* out, struct CUstream_st* stream) {
    if (!in || !out || n == 0 || k < 1 || (size_t)k > n) return TOPK_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 3u) return TOPK_ERR_INVALID_ARG;
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
    if (a < b + (size_t)k * sizeof(int32_t) && b < a + n * sizeof(int32_t)) return TOPK_ERR_INVALID_ARG;
    if (k > TOPK_NOALLOC_MAX_K || n > (size_t(1) << 40)) return TOPK_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) {
        topk::note_cuda_error((int)e);
        return TOPK_ERR_CUDA;
    }
    // No staging here: both buffers must already be in device memory.
    if (!is_device_memory(in) || !is_device_memory(out)) return TOPK_ERR_INVALID_ARG;

    void* scratch = nullptr;
    int rc = scratch_address(device, &scratch);
    if (rc != TOPK_OK) return rc;

    if (k > 128) {
        // Large k: radix select, its candidate buffer sized to what the
        // array leaves after the control words and the histogram.
        const size_t cap = kNoallocRadixCap;
        int launches = 0;
        e = cudaMemsetAsync(static_cast<char*>(scratch) + topk::kI32ResetBegin, 0,
                            topk::kI32ResetEnd - topk::kI32ResetBegin, s);
        topk::note_unreleased_launch(device, s);
        if (e == cudaSuccess) e = topk::radix_launch(s, in, n, k, out, scratch, cap, &launches, false);
        for (int i = 0; i < launches; ++i) topk::note_launch();
        if (e != cudaSuccess) {
            topk::note_cuda_error((int)e);
            return TOPK_ERR_CUDA;
        }
        return TOPK_OK;
    }

    topk::I32Plan plan;
    e = topk::i32_plan(device, n, k, &plan);
    if (e != cudaSuccess) {
        topk::note_cuda_error((int)e);
        return TOPK_ERR_CUDA;
    }
    // Fewer blocks when the candidates of a full grid would not fit; the
    // kernel's grid-stride loop covers the input with any grid size.
    const size_t fit = (kNoallocScratchBytes - topk::kI32CandOffset) / (topk::kI32CandPerBlock * sizeof(int32_t));
    if ((size_t)plan.grid > fit) plan.grid = (int)fit;

    // The array keeps the last call's contents; the control words and the
    // block-maximum slots must start at zero, so clear them on the stream
    // before the launch (the sticky status word is left alone).
    e = cudaMemsetAsync(static_cast<char*>(scratch) + topk::kI32ResetBegin, 0,
                        topk::kI32ResetEnd - topk::kI32ResetBegin, s);
    // A launch of this library that follows on the stream must not start
    // early: it may read this call's output.
    topk::note_unreleased_launch(device, s);
    if (e == cudaSuccess) e = topk::i32_launch(plan, s, in, n, k, out, scratch, false, false);
    if (e != cudaSuccess) {
        topk::note_cuda_error((int)e);
        return TOPK_ERR_CUDA;
    }
    topk::note_launch();
    return TOPK_OK;
}
