/*
 * topk.h -- C ABI of libtopk.so, TopK selection on one NVIDIA GB300 (sm_103a).
 *
 * Two operations, both from "CUDA parallel optimisation: TopK, shared memory
 * and two-stage reduction":
 *
 *   topk_i32       the k largest values of an int32 array, sorted descending
 *                  (sections 2.1-2.2: a block-level pass that leaves k
 *                  candidates per block, then a second pass over the
 *                  candidates; the result equals the CPU's exactly).
 *   topk_rows_f32  per row of a float32 matrix, the k best scores with their
 *                  column indices (section 6, update_candidates: TopK keyed
 *                  by a score that carries an item id).
 *
 * Conventions shared by every entry point:
 *   - Pointers may be device memory (cudaMalloc, managed) or host memory
 *     (pageable or pinned).  The library asks the CUDA runtime which one it
 *     is.  Device pointers: the call only enqueues work on `stream` and
 *     returns; read the outputs after synchronising the stream.  If any
 *     pointer is host memory: inputs are copied to device staging, outputs
 *     are copied back, and the call returns only after `stream` has
 *     finished, so host outputs are ready on return.
 *   - `stream` is a cudaStream_t; NULL means the legacy default stream.
 *   - Inputs are read-only.  Outputs must not overlap inputs.  Any 4-byte
 *     aligned address is accepted.
 *   - The caller owns every buffer it passes.  The library owns a cached
 *     device workspace per (device, stream), grown on demand with
 *     cudaMalloc and freed by topk_release_workspace().  Calls on one stream
 *     share that stream's workspace in stream order; calls on different
 *     streams never share one.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and leave the outputs untouched.
 *   - The current CUDA device is the one used.
 */
#ifndef TOPK_GB300_TOPK_H
#define TOPK_GB300_TOPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

/* Status codes returned by every entry point. */
enum topk_status {
    TOPK_OK = 0,
    TOPK_ERR_INVALID_ARG = 1, /* null pointer, n == 0, k < 1, k > n, rows < 1, cols < k, overlap */
    TOPK_ERR_UNSUPPORTED = 2, /* k above TOPK_MAX_K / TOPK_MAX_K_ROWS, or a size the kernels do not take */
    TOPK_ERR_NO_MEMORY = 3,   /* workspace or staging allocation failed */
    TOPK_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed; see topk_last_cuda_error() */
    TOPK_ERR_DEVICE_TIMEOUT = 5 /* a kernel's bounded wait gave up; its results are not valid */
};

/* Largest k accepted by topk_i32, topk_u32 and topk_f32. */
#define TOPK_MAX_K 131072

/* Largest k accepted by topk_i32_noalloc. */
#define TOPK_NOALLOC_MAX_K 32768

/* Largest k accepted by topk_rows_f32. */
#define TOPK_MAX_K_ROWS 1024

/*
 * topk_i32 -- the k largest values of in[0..n), written to out[0..k) in
 * descending order.  Equal values appear as often as they occur in the input
 * (the result is a multiset; there are no indices, so no tie order).
 *
 *   in     int32[n], read-only.
 *   n      number of elements, 1 <= n <= 2^40.
 *   k      1 <= k <= min(n, TOPK_MAX_K).
 *   out    int32[k], written.
 *
 * k <= 128: one launch.  Every block filters its share of the input against
 * a running k-th-value threshold and leaves k candidates; the last block to
 * finish merges the candidates (section 2.2's second pass, fused into the
 * same launch).  k > 128: a radix select on order-preserving keys ("GPU
 * radix sort", histogram section).  When n exceeds 2^18, a threshold is
 * taken from a 2^16-key sample, one pass over the input keeps the keys above
 * it, and one 8-CTA cluster selects the k-th key among them and sorts the
 * answer (five launches, one input pass; two or three more input passes
 * run, inside one of those launches, only when the sample misled the
 * filter).  When n <= 2^18 the cluster does it all in
 * one launch.  k > 32768: the cluster leaves the answer unordered and the
 * library's LSD radix sort (topk_sort_u32's kernels) orders it, plus one
 * launch that writes it out; that form needs about 4k more bytes of
 * workspace and sort scratch for k keys.
 *
 * Returns TOPK_OK or an error code; on error nothing is written to out.
 */
int topk_i32(const int32_t* in, size_t n, int k, int32_t* out, struct CUstream_st* stream);

/*
 * topk_u32 -- topk_i32 for uint32 keys: the k largest of in[0..n) in
 * unsigned order, descending ("GPU radix sort" sorts uint32 keys; the TopK
 * of sections 2.1-2.2 on them).  Arguments, limits, plans and errors are
 * those of topk_i32.
 *
 * topk_f32 -- topk_i32 for float32 keys: the k largest of in[0..n) under
 * IEEE 754 totalOrder, descending, each output the bits of an input
 * element.  totalOrder is the order the "GPU radix sort" page gives floats
 * with its bit transform (extensions section): -NaN < -inf < ... < -0.0 <
 * +0.0 < ... < +inf < +NaN, NaNs of one sign ordered by payload (larger
 * payloads further from zero).  So every bit pattern is its own key: -0.0
 * ranks below +0.0, and a NaN with the sign bit set ranks below -inf.
 * Arguments, limits, plans and errors are those of topk_i32.
 */
int topk_u32(const uint32_t* in, size_t n, int k, uint32_t* out, struct CUstream_st* stream);
int topk_f32(const float* in, size_t n, int k, float* out, struct CUstream_st* stream);

/*
 * topk_rows_f32 -- for each row r of the row-major rows x cols matrix `in`,
 * the k best entries: vals[r*k + j] is the j-th best value of row r and
 * idx[r*k + j] its column.
 *
 * Order: value descending; among equal values the lower column index comes
 * first.  -0.0 and +0.0 are equal.  NaN ranks above +inf and all NaNs are
 * equal (so among NaNs the lower column wins).  Values are copied bit for bit
 * from the input (a -0.0 stays -0.0, a NaN keeps its payload).
 *
 *   in     float32[rows * cols], row-major, read-only.
 *   rows   1 <= rows <= 2^31 - 1.
 *   cols   k <= cols <= 2^31 - 1.
 *   k      1 <= k <= min(cols, TOPK_MAX_K_ROWS).
 *   vals   float32[rows * k], written.
 *   idx    int32[rows * k], written.
 *
 * Returns TOPK_OK or an error code; on error nothing is written.
 */
int topk_rows_f32(const float* in, int rows, int cols, int k, float* vals, int32_t* idx,
                  struct CUstream_st* stream);

/*
 * topk_items_f32 -- score-keyed TopK with item ids, with an optional filter
 * in front ("CUDA parallel optimisation: TopK ...", section 6:
 * update_candidates(candidates, k, item, score), and its remark that stages
 * compose: filter first, then TopK; merge several TopK results).
 *
 * Among the positions i of score[0..n) with keep[i] != 0 (every position
 * when keep is null), the k best: score descending, NaN above +inf, -0.0
 * equal to +0.0, the lower position first among equal scores -- the order
 * of topk_rows_f32.  out_score[j] is the j-th best score (the input's bits),
 * out_item[j] its item: item[i], or the position i when item is null.  When
 * fewer than k positions are kept, the remaining entries hold -inf and item
 * -1, and *out_count (if out_count is not null) is the number of real
 * entries.  Merging several TopK results is this call on their
 * concatenated scores and items.
 *
 *   score      float32[n], device memory.
 *   item       int64[n] or null, device memory.
 *   keep       uint8[n] or null, device memory (nonzero = candidate).
 *   n          1 <= n <= 2^31 - 1.
 *   k          1 <= k <= min(n, TOPK_MAX_K_ROWS).
 *   out_score  float32[k]; out_item int64[k]; out_count one int64 or null.
 *
 * The selection is a two-stage reduction applied level by level: rows of at
 * least 8k scores give their k best (the row TopK), and their winners, in
 * order, are the next level's candidates (blocks of 1024 keeping their k
 * best for k <= 128, rows again otherwise) until one block ranks the last
 * at most 4096.  With keep, when
 * n >= 2^20, k <= 128 and keep's address is congruent to score's / 4
 * (mod 4) (e.g. score 16-byte aligned, keep 4-byte aligned), the first
 * level skips filtered positions itself and the call only enqueues.
 * Otherwise an ordered compaction of the kept scores runs first, and the
 * call waits for the kept count (a 4-byte copy to the host) before it
 * enqueues the levels; that form needs about 8n bytes more scratch.  Without
 * keep the call only enqueues.  Scratch: about 24 * 4097 * k bytes besides,
 * in the library's per-stream workspace.
 * Host pointers are rejected with TOPK_ERR_INVALID_ARG.
 */
int topk_items_f32(const float* score, const int64_t* item, const uint8_t* keep, size_t n, int k, float* out_score,
                   int64_t* out_item, int64_t* out_count, struct CUstream_st* stream);

/*
 * topk_sort_u32 -- sort n uint32 keys ascending, stably, carrying uint32
 * values if given: an LSD radix sort with 8-bit digits, four passes ("GPU
 * radix sort": sections 2-4; key-value pairs from its extensions section).
 * Equal keys keep their input order, and each value travels with its key.
 *
 *   keys       uint32[n], device memory, read-only.
 *   vals       uint32[n] or null (keys only), device memory, read-only.
 *   n          1 <= n <= 2^32 - 1.
 *   keys_out   uint32[n], device memory, written; must not overlap the inputs.
 *   vals_out   uint32[n], written; null exactly when vals is null.
 *
 * Five launches: one histogram pass for all four digits, then one pass per
 * digit in which every 8192-key tile ranks its keys, finds where its keys of
 * each digit go from the tiles before it (decoupled look-back, bounded
 * waits) and writes them in digit order.  Scratch (in the library's
 * per-stream workspace): about 4n bytes (8n with values) plus 0.5 byte per
 * key of look-back words.  The call only enqueues work.  Host pointers are
 * rejected with TOPK_ERR_INVALID_ARG.
 */
int topk_sort_u32(const uint32_t* keys, const uint32_t* vals, size_t n, uint32_t* keys_out, uint32_t* vals_out,
                  struct CUstream_st* stream);

/* Operations of topk_reduce_i32 / topk_reduce_f32. */
enum topk_reduce_op { TOPK_REDUCE_SUM = 0, TOPK_REDUCE_MAX = 1, TOPK_REDUCE_MIN = 2 };

/*
 * topk_reduce_i32 / topk_reduce_f32 -- the sum, maximum or minimum of
 * in[0..n), in one launch: the two-stage block/warp reduction of "CUDA
 * reduction, complete guide" (its warp-shuffle level and multi-level
 * system), which the TopK page (section 6) names as the same pattern as the
 * TopK.  Every block reduces its share to one partial; the last block to
 * finish reduces the partials.
 *
 *   in     int32[n] or float32[n], read-only; any 4-byte-aligned address.
 *   n      1 <= n <= 2^40.
 *   op     TOPK_REDUCE_SUM, TOPK_REDUCE_MAX or TOPK_REDUCE_MIN.
 *   out    one int64_t (int32 input) or one double (float32 input), written;
 *          8-byte aligned.
 *
 * int32: the sum is exact (int64, no wrap); max and min are widened to int64.
 * float32 max/min: IEEE 754-2019 maximum/minimum -- any NaN gives the
 *   canonical quiet NaN, and -0.0 counts as below +0.0; exact.
 * float32 sum: pairwise float32 sums of 4, added with compensation over
 *   batches of 32 elements and folded into doubles; the result is within
 *   2^-22 * sum|x| (plus double rounding) of the exact sum.  +inf, -inf and NaN propagate as in IEEE arithmetic.
 *   A batch whose float partial sum passes FLT_MAX (inputs near 1e37 and
 *   above) gives inf.
 * Pointers may be device or host memory, as for topk_i32.
 * Returns TOPK_OK or an error code (TOPK_ERR_INVALID_ARG for a null pointer,
 * n == 0, an unknown op or misalignment); on error out is not written.
 */
int topk_reduce_i32(const int32_t* in, size_t n, int op, int64_t* out, struct CUstream_st* stream);
int topk_reduce_f32(const float* in, size_t n, int op, double* out, struct CUstream_st* stream);

/* Bytes of the device array that topk_i32_noalloc uses as scratch. */
#define TOPK_NOALLOC_SCRATCH_BYTES (1u << 20)

/*
 * topk_i32_noalloc -- topk_i32 without any allocation.  The pages have no
 * counterpart; it exists for callers that cannot call cudaMalloc: the
 * enqueue hook of a framework plugin that is not allowed to allocate, a
 * process whose device memory is already claimed by another allocator's
 * pool, or a latency-bound loop that cannot take the implicit
 * synchronisation of cudaMalloc/cudaFree.
 *
 * Same arguments, result and errors as topk_i32, except:
 *   - in and out must be device (or managed) memory; host pointers are
 *     rejected with TOPK_ERR_INVALID_ARG (staging them would allocate).
 *   - The scratch is one file-scope device array of
 *     TOPK_NOALLOC_SCRATCH_BYTES (1 MiB): control words, per-block maxima
 *     and per-block candidates.  Every GPU that loads the library holds it
 *     until the process exits.  k above TOPK_NOALLOC_MAX_K is rejected with
 *     TOPK_ERR_UNSUPPORTED.  For k <= 128 the grid is cut so that every
 *     block's candidate lists fit (1 MiB holds 239 blocks' worth), so on
 *     GPUs with more SMs this entry point runs fewer blocks than topk_i32;
 *     for larger k the radix select's candidate buffer is what the array
 *     has left (252,800 keys instead of 262,144), so slightly fewer inputs
 *     avoid the exact passes.
 *   - Every call uses the same array.  Each call clears the control words
 *     on `stream` before its launch, but calls whose work overlaps on the
 *     GPU (different streams, or different host threads without ordering)
 *     race on the array and may return wrong results.  Order them.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - No cudaMalloc, cudaFree or other allocating call is made.
 */
int topk_i32_noalloc(const int32_t* in, size_t n, int k, int32_t* out, struct CUstream_st* stream);

/*
 * topk_check_stream -- wait for `stream`, then report whether any TopK
 * kernel that ran on it (through that stream's workspace, or through
 * topk_i32_noalloc on the current device) gave up on a device-side wait.
 * The kernels never spin without limit: each wait on another warp's
 * progress stops after a fixed number of tries, sets a sticky status word
 * and lets the launch finish, leaving invalid results.  This call reads and
 * clears that word.  Returns TOPK_OK, TOPK_ERR_DEVICE_TIMEOUT or
 * TOPK_ERR_CUDA.
 *
 * topk_i32_noalloc has one status word per device, shared by every stream:
 * a timeout of a no-alloc call on another stream is reported to whichever
 * caller checks first, and one set while this call runs may be missed.
 * Synchronise the device first when that matters.
 */
int topk_check_stream(struct CUstream_st* stream);

/* Options for topk_set_option. */
enum topk_option {
    /* Upper bound on the number of candidates the int32 second stage sorts
     * in shared memory (a power of two >= 2; 0 restores the default, which
     * is what fits).  When more candidates exceed the final threshold, the
     * second stage first finds the exact k-th value by radix select.  Lower
     * it only to exercise that path; results are the same either way. */
    TOPK_OPT_STAGE2_CAP = 1,
    /* Upper bound, in keys, on the candidate buffer of the large-k plan
     * (k > 128; 0 restores the default; values below k act as k).  Inputs
     * whose candidates overflow it take the exact radix passes.  Lower it
     * only to exercise those passes; results are the same either way. */
    TOPK_OPT_RADIX_CAP = 2,
    /* Rank, within the large-k plan's 2^16-key sample, of the key used as
     * the filter threshold (0 restores the automatic choice).  A rank that
     * is too small makes the filter keep fewer than k keys, and the plan
     * takes the exact radix passes.  For tests of that path only. */
    TOPK_OPT_RADIX_SAMPLE_RANK = 3,
    /* Share of the input tiles that topk_i32's streaming plan (k <= 128)
     * assigns to warps up front, as percent + 1 (1 = none, 101 = all; 0
     * restores the default).  The other tiles are claimed one at a time
     * from counters as warps finish, so that fast SMs take the slow ones'
     * share.  For tests of both schedules; results are the same either way. */
    TOPK_OPT_STREAM_STATIC = 4,
    /* 1: no call starts early (see topk_last_launch_early); every launch
     * waits for the previous work on its stream.  0 (the default): early
     * start as described there.  Set it when work that is not this
     * library's writes a TopK input on the same stream between two calls
     * and must be finished, memory flushed, before the next call reads. */
    TOPK_OPT_NO_EARLY_START = 5,
    /* 1: every later workspace or staging allocation fails with
     * TOPK_ERR_NO_MEMORY, as if the device were full; 0: normal.  The
     * environment variable TOPK_FAULT_ALLOC=1, read at the first
     * allocation, sets it too.  For tests of callers' error paths (the
     * failure is made on the host; no device fault). */
    TOPK_OPT_FAULT_ALLOC = 6,
    /* Polls of one look-back word before a tile of topk_sort_u32 gives up
     * (0 restores the default, 2^22).  A tile that gives up writes its keys
     * to wrong places inside the output (never outside it), and
     * topk_check_stream then reports TOPK_ERR_DEVICE_TIMEOUT.  Lower it
     * only to exercise that report. */
    TOPK_OPT_SORT_SPINS = 7,
    /* 1: the first tile of every digit pass of topk_sort_u32 withholds its
     * look-back word (0 restores the default).  The tile after it then
     * polls a word that nothing writes until the poll limit runs out, gives
     * up, and topk_check_stream reports TOPK_ERR_DEVICE_TIMEOUT; the output
     * is then wrong but every write stays inside it.  Only to exercise that
     * report, with TOPK_OPT_SORT_SPINS lowered so that the wait is short. */
    TOPK_OPT_SORT_WITHHOLD = 8
};

/* Set a process-wide option; takes effect for calls made afterwards.
 * Returns TOPK_OK or TOPK_ERR_INVALID_ARG. */
int topk_set_option(int option, int value);

/* A static, human-readable name for a status code. */
const char* topk_status_string(int status);

/* The cudaError_t value behind the last TOPK_ERR_CUDA returned on the
 * calling thread (0 if none). */
int topk_last_cuda_error(void);

/* Free every cached workspace of the calling process (all devices, all
 * streams).  The caller must make sure no TopK work is still running.
 * Workspaces are kept per (device, stream handle) and are not dropped when a
 * stream is destroyed, so a program that creates and destroys streams in a
 * loop should call this now and then.  Returns TOPK_OK or TOPK_ERR_CUDA. */
int topk_release_workspace(void);

/* Whether the last TopK launch this thread enqueued may start while the
 * previous kernel on its stream finishes (1) or waits for it (0); a
 * diagnostic for tests of the early-start rule below.
 *
 * Early start: the streaming kernels of topk_i32 (k <= 128) and
 * topk_rows_f32 (k <= 128) are launched with programmatic stream
 * serialization.  When the previous kernel on the stream is one of those
 * launches (or the last kernel of topk_i32's large-k plan), the new call
 * begins reading its input while that launch finishes, provided the input
 * does not overlap what that launch writes; everything else the call
 * touches waits for it.  Every other entry point, and a call whose buffers
 * are host memory, resets this, so the call after it starts normally. */
int topk_last_launch_early(void);

/* Number of CUDA kernels this library has launched in this process; a
 * diagnostic for benchmarks that count launches. */
unsigned long long topk_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* TOPK_GB300_TOPK_H */
