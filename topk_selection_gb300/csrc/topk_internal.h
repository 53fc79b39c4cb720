// Declarations shared between the C ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace topk {

// Control words of one int32 TopK launch.  Both are zero between launches:
// the last block of a launch resets them after use.
//   thresh  the largest published threshold, stored as (value ^ 0x80000000)
//           so that unsigned order is signed order and 0 means INT_MIN.
//   ticket  number of blocks that have finished stage 1.
struct I32Ctrl {
    unsigned thresh;
    unsigned ticket;
    unsigned pad[62];  // one 256-byte line to itself
};

struct I32Plan {
    int grid;      // blocks launched
    int max_grid;  // persistent grid size for this device (blocks per SM x SMs)
};

// Grid for an n-element, k-wide selection on `device`.
cudaError_t i32_plan(int device, size_t n, int k, I32Plan* plan);

// Enqueue the single-launch int32 TopK.  cand holds plan.grid * k ints;
// ctrl must be zero (it is again when the launch completes).
cudaError_t i32_launch(const I32Plan& plan, cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out,
                       int32_t* cand, I32Ctrl* ctrl);

// Enqueue the row TopK (one block per row).
cudaError_t rows_launch(cudaStream_t s, const float* in, int rows, int cols, int k, float* vals, int32_t* idx);

// Bookkeeping of the C ABI layer, for entry points defined in other files:
// record the cudaError_t behind a TOPK_ERR_CUDA, and count a kernel launch.
void note_cuda_error(int err);
void note_launch();

}  // namespace topk
