// Declarations shared between the C ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace topk {

// Key kinds of the 32-bit TopK entry points: int32 (topk_i32), uint32
// (topk_u32) and float32 bit patterns under IEEE 754 totalOrder (topk_f32).
enum KeyKind : int { kKeyI32 = 0, kKeyU32 = 1, kKeyF32 = 2 };

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

// Scratch of an int32 TopK launch.  Both plans (streaming, k <= 128; radix
// select, larger k) use the same workspace, laid out so that every byte one
// of them needs zero at its start is one that both leave zero at their end:
//   [0, 256)                     status word: nonzero after a bounded wait gave
//                                up (sticky; read and cleared by the host)
//   [256, 512)                   control words: I32Ctrl (streaming) or the
//                                radix control words
//   [512, 512 + 8*4096)          streaming: per-block running maxima (first
//                                4 KiB), then the tile-claim counters (64 x
//                                128 bytes); radix: the global 12-bit digit
//                                histogram (64-bit counts)
//   -- everything above is zero between launches: [kI32ResetBegin, kI32ResetEnd) --
//   [kRadixCandOffset, +4096)    radix: the range table the cluster kernel
//                                leaves for the sort kernel
//   [kRadixBufOffset, ...)       radix: the candidate buffer (cap keys)
//   [kI32CountOffset, +4*8192)   streaming: per-list survivor counts (the
//                                first 1024), then tile maxima (1024)
//   [kI32CandOffset, ...)        streaming: per block, its candidate lists
//                                (up to kI32CandPerBlock ints)
// The last two areas overlap the radix buffer; none of them needs any value
// at the start of a launch.
constexpr int kI32MaxGrid = 1024;
constexpr int kI32MaxListsPerBlock = 8;
constexpr int kI32CandPerBlock = 1024;
constexpr size_t kI32StatusOffset = 0;
constexpr size_t kI32CtrlOffset = 256;
constexpr size_t kI32BmaxOffset = 512;
constexpr size_t kRadixCtrlOffset = kI32CtrlOffset;
constexpr size_t kRadixHistOffset = kI32BmaxOffset;
constexpr size_t kRadixCandOffset = kRadixHistOffset + 4096 * sizeof(unsigned long long);
constexpr size_t kRadixPlanBytes = 4096;
constexpr size_t kRadixBufOffset = kRadixCandOffset + kRadixPlanBytes;
constexpr size_t kI32ResetBegin = kI32CtrlOffset;
constexpr size_t kI32ResetEnd = kRadixCandOffset;
constexpr size_t kI32CountOffset = kRadixCandOffset;
constexpr size_t kI32CandOffset =
    kI32CountOffset + (size_t)kI32MaxGrid * kI32MaxListsPerBlock * sizeof(int32_t);
constexpr int kRadixMaxK = 32768;
static_assert(kI32BmaxOffset + kI32MaxGrid * sizeof(unsigned) <= kI32ResetEnd, "block maxima are reset");
// Streaming plan: the tile-claim counters of the dynamic part of the
// schedule, one per 128-byte line (zero between launches), ...
constexpr int kI32DynRanges = 64;  // two warp-wide words of ballots
constexpr size_t kI32DynStride = 128;
constexpr size_t kI32DynOffset = kI32BmaxOffset + kI32MaxGrid * sizeof(unsigned);
static_assert(kI32DynOffset + kI32DynRanges * kI32DynStride <= kI32ResetEnd, "claim counters are reset");
// ... and, when the grid has fewer blocks than k, every tile's maximum
// (written before it is read; at most kI32MaxTileMax tiles), after the
// per-list counts of kI32MaxGrid lists.
constexpr int kI32MaxTileMax = 1024;
constexpr size_t kI32TileMaxOffset = kI32ResetEnd + (size_t)kI32MaxGrid * sizeof(int32_t);
static_assert(kI32TileMaxOffset + kI32MaxTileMax * sizeof(int32_t) <=
                  kI32ResetEnd + (size_t)kI32MaxGrid * kI32MaxListsPerBlock * sizeof(int32_t),
              "tile maxima sit in the unused part of the per-list counts");
static_assert(kRadixCandOffset % 256 == 0 && kRadixBufOffset % 256 == 0 && kI32CountOffset % 256 == 0 &&
                  kI32CandOffset % 256 == 0,
              "area alignment");

// Keys one thread-block cluster of the radix plan holds in shared memory
// (8 CTAs x 32768); the candidate buffer never exceeds it.
constexpr size_t kRadixClusterCap = size_t(1) << 18;
// Candidate buffer of the radix plan in the cached workspace, in keys.
constexpr size_t kRadixCap = kRadixClusterCap;

constexpr size_t radix_scratch_bytes(size_t cap) { return kRadixBufOffset + cap * sizeof(unsigned); }

// Enqueue the radix-select int32 TopK (two launches when n fits one
// cluster, else seven; any k up to kRadixMaxK).  scratch holds radix_scratch_bytes(cap)
// bytes, 256-byte aligned, whose [kI32ResetBegin, kI32ResetEnd) bytes are
// zero (they are zero again afterwards); cap is the candidate buffer's
// capacity in keys, k <= cap <= kRadixClusterCap.  Every kernel of the plan
// waits for its predecessor's writes before reading anything.  release: the
// plan's last kernel lets the next launch on the stream start before it
// completes; only for callers that make sure such a launch does not read
// `out` before it waits (see i32_launch's `early`).
// kind: the key kind (0 int32, 1 uint32, 2 float32 under totalOrder).
// bigk: null, or (for k above kRadixMaxK) k words where the plan leaves the
// complements of the TopK's keys, unordered, instead of sorting them into
// `out`: the caller sorts them ascending (sort_launch) and writes `out` with
// radix_bigk_out.
cudaError_t radix_launch(cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out, void* scratch,
                         size_t cap, int* launches, bool release, int kind = 0, uint32_t* bigk = nullptr);
cudaError_t radix_bigk_out(cudaStream_t s, const uint32_t* sorted, int k, int32_t* out, int kind);
// Largest k of the big-k form (a share of the candidate buffer, so that the
// sampled threshold usually keeps few enough candidates).
constexpr int kBigKMax = 131072;
static_assert(kBigKMax * 2 <= (int)kRadixCap, "the big-k form keeps half the candidate buffer free");

// Test options of the radix plan (TOPK_OPT_RADIX_CAP, TOPK_OPT_RADIX_SAMPLE_RANK; 0 = default).
int radix_cap_option();
int radix_sample_rank_option();

// Status bits a kernel may set in the status word.
constexpr unsigned kStatusWaitTimeout = 1u;

constexpr size_t i32_scratch_bytes(int grid) {
    return kI32CandOffset + (size_t)grid * kI32CandPerBlock * sizeof(int32_t);
}

struct I32Plan {
    int grid;        // blocks launched (<= kI32MaxGrid)
    int max_grid;    // persistent grid size for this device (blocks per SM x SMs), <= kI32MaxGrid
    int stage2_cap;  // 0, or a lower capacity for the second stage's shared list (TOPK_OPT_STAGE2_CAP)
    int static_pct;  // share of the tiles, in percent, assigned statically; the rest are claimed
    int kind;        // key kind (KeyKind of topk_device.cuh): int32, uint32 or float32 words
};

// Current value of TOPK_OPT_STAGE2_CAP (0 = default).
int stage2_cap_option();
// Current value of TOPK_OPT_STREAM_STATIC (0 = default, else percent + 1).
int stream_static_option();
// Current value of TOPK_OPT_SORT_SPINS (0 = default).
int sort_spins_option();

// Grid for an n-element, k-wide selection on `device` (k <= 128: the
// streaming plan; larger k use radix_launch).
// kind: the key kind (0 int32, 1 uint32, 2 float32 under totalOrder).
cudaError_t i32_plan(int device, size_t n, int k, I32Plan* plan, int kind = 0);

// Enqueue the single-launch int32 TopK.  scratch holds i32_scratch_bytes(plan.grid)
// bytes, 256-byte aligned, whose [kI32ResetBegin, kI32ResetEnd) bytes are zero
// (they are zero again when the launch completes).  early: launch with
// programmatic stream serialization, so that when the previous kernel on the
// stream released its successors early (see `release`), this launch starts
// streaming its input while that one finishes; the input must then not be
// anything the previous launch writes (its output).  release: once its
// blocks have read their input, let the next launch start early; only for
// callers that record this launch's output for that check.
cudaError_t i32_launch(const I32Plan& plan, cudaStream_t s, const int32_t* in, size_t n, int k, int32_t* out,
                       void* scratch, bool early, bool release);

// Enqueue the row TopK.  status: a device word that bounded waits set to
// kStatusWaitTimeout when they give up (sticky).  For k <= 128: early
// launches with programmatic stream serialization, so the kernel may start
// while the previous kernel on the stream finishes; flags:
//   kRowsRelease    let the next launch start early (as i32_launch's release);
//   kRowsWaitFirst  wait for the previous kernel before reading the input
//                   (its input is that kernel's output); without it an early
//                   launch reads its input first, so the input must not
//                   overlap what the previous launch writes.
constexpr int kRowsRelease = 1, kRowsWaitFirst = 2;
cudaError_t rows_launch(cudaStream_t s, const float* in, int rows, int cols, int k, float* vals, int32_t* idx,
                        unsigned* status, bool early, int flags);

// The row TopK over kept elements only (k <= 128): element (r, c) takes part
// when keep[r * cols + c] != 0.  Each row's outputs hold its valid winners
// first, then (-inf, -1); row_count[r] is how many are valid.  Needs
// rows_mask_aligned(in, keep) (cudaErrorInvalidValue otherwise).
bool rows_mask_aligned(const float* in, const uint8_t* keep);
cudaError_t rows_launch_masked(cudaStream_t s, const float* in, const uint8_t* keep, int rows, int cols, int k,
                               float* vals, int32_t* idx, int32_t* row_count, unsigned* status, bool early,
                               int flags);

// Enqueue a one-launch reduction (op 0 sum, 1 max, 2 min) of n int32 or
// float32 values.  out: one int64 (int32 input) or one double (float32
// input), in device memory.  scratch: the int32 workspace (its ticket word in
// the control line is zero and is left zero; block partials go after the
// control area, 32 bytes per block, at most kI32MaxGrid blocks).
cudaError_t reduce_launch(cudaStream_t s, const void* in, size_t n, bool is_float, int op, void* out, void* scratch);
constexpr size_t kReduceScratchBytes = kI32CandOffset + (size_t)kI32MaxGrid * 32;

// Score-keyed TopK with item ids and an optional keep filter (topk_items.cu).
// scratch: items_scratch_bytes(n, k, compact) bytes of device memory, compact
// = keep != null && !items_fused_filter(score, keep, n, k)
// (no contents needed).  With a filter that does not fold into the first
// level, the call waits for the kept count (one 4-byte copy to the host)
// before enqueueing the selection.
// compact: the filter runs as a separate compaction (a keep array that
// items_fused_filter turns down); its arrays need n * 8 more bytes.
size_t items_scratch_bytes(size_t n, int k, bool compact);
// Whether a filtered call folds the filter into its first level (no
// compaction, no wait for the kept count).
bool items_fused_filter(const float* score, const uint8_t* keep, size_t n, int k);
cudaError_t items_launch(cudaStream_t s, const float* score, const int64_t* item, const uint8_t* keep, size_t n,
                         int k, float* out_score, int64_t* out_item, int64_t* out_count, void* scratch,
                         size_t scratch_bytes, unsigned* status, int* launches);

// LSD radix sort of uint32 keys (optionally with uint32 values), stable,
// ascending (topk_sort.cu).  scratch: sort_scratch_bytes(n, vals != null)
// bytes whose first kSortHeaderBytes are zero before the first call on it
// (the kernels leave them so); epoch: a number that differs between calls
// on the same scratch (it tags the look-back words).  n < 2^32.
constexpr size_t kSortHeaderBytes = 16384;
size_t sort_scratch_bytes(size_t n, bool with_vals);
cudaError_t sort_launch(cudaStream_t s, const uint32_t* keys, const uint32_t* vals, size_t n, uint32_t* keys_out,
                        uint32_t* vals_out, void* scratch, unsigned epoch, unsigned* status, int* launches);

// Bookkeeping of the C ABI layer, for entry points defined in other files:
// record the cudaError_t behind a TOPK_ERR_CUDA, and count a kernel launch.
void note_cuda_error(int err);
void note_launch();

// Device address of topk_i32_noalloc's scratch on `device`, or null if that
// entry point has not run there yet.
void* noalloc_scratch_if_ready(int device);

// Record, for entry points without a cached workspace, that the last launch
// on stream s of `device` does not let its successor start early (so the
// next launch there does not start early either).
void note_unreleased_launch(int device, cudaStream_t s);

}  // namespace topk
