/*
 * Seeded synthetic inputs for the TopK workloads.
 *
 * This module only draws numbers; it holds none of the selection arithmetic.
 * Both the CPU oracle and the CUDA path read the buffers it fills, so the
 * two sides always see the same bytes.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; the 64-bit finaliser constants are the
 * ones Vigna publishes with splitmix64.c).  The i-th output of a SplitMix64
 * stream seeded with s is mix(s + (i + 1) * golden_gamma), so any element can
 * be computed from its index alone and large arrays are filled in parallel.
 *
 * Workloads (from the configurations the TopK pages benchmark):
 *   - int32 uniform over the full range: (int32)(uint32)(x_i >> 32)
 *   - int32 heavy duplicates in [0, m): x_i % m
 *   - int32 sorted ascending: in[i] = i
 *   - float32 N(0,1): Box-Muller in double on the pair (x_2p, x_2p+1)
 *   - tie forcing: per row, m distinct positions (partial Fisher-Yates on a
 *     per-row stream) are overwritten with that row's maximum
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL
#define ROW_STREAM_SALT 0xD1B54A32D192ED03ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* i-th output (0-based) of the SplitMix64 stream seeded with `seed`. */
uint64_t synth_splitmix64_at(uint64_t seed, uint64_t i) {
    return mix64(seed + (i + 1) * GOLDEN_GAMMA);
}

/* ---- a tiny parallel-for over [0, n) ---------------------------------- */

typedef void (*range_fn)(void* ctx, size_t lo, size_t hi);

typedef struct {
    range_fn fn;
    void* ctx;
    size_t lo, hi;
} range_job;

static void* run_range(void* p) {
    range_job* j = (range_job*)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

static void parallel_for(size_t n, int nthreads, range_fn fn, void* ctx, size_t min_per_thread) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((size_t)nthreads > n / min_per_thread + 1) nthreads = (int)(n / min_per_thread + 1);
    if (nthreads == 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t tid[256];
    range_job jobs[256];
    int started[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].lo = n * (size_t)t / (size_t)nthreads;
        jobs[t].hi = n * (size_t)(t + 1) / (size_t)nthreads;
        started[t] = pthread_create(&tid[t], NULL, run_range, &jobs[t]) == 0;
        if (!started[t]) run_range(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (started[t]) pthread_join(tid[t], NULL);
}

/* ---- int32 workloads --------------------------------------------------- */

typedef struct {
    int32_t* out;
    uint64_t seed;
    uint32_t m;
} i32_ctx;

static void fill_uniform(void* p, size_t lo, size_t hi) {
    i32_ctx* c = (i32_ctx*)p;
    for (size_t i = lo; i < hi; ++i)
        c->out[i] = (int32_t)(uint32_t)(synth_splitmix64_at(c->seed, i) >> 32);
}

static void fill_mod(void* p, size_t lo, size_t hi) {
    i32_ctx* c = (i32_ctx*)p;
    for (size_t i = lo; i < hi; ++i)
        c->out[i] = (int32_t)(synth_splitmix64_at(c->seed, i) % c->m);
}

static void fill_ascending(void* p, size_t lo, size_t hi) {
    i32_ctx* c = (i32_ctx*)p;
    for (size_t i = lo; i < hi; ++i) c->out[i] = (int32_t)(uint32_t)i;
}

void synth_i32_uniform(int32_t* out, size_t n, uint64_t seed, int nthreads) {
    i32_ctx c = {out, seed, 0};
    parallel_for(n, nthreads, fill_uniform, &c, 65536);
}

void synth_i32_mod(int32_t* out, size_t n, uint64_t seed, uint32_t m, int nthreads) {
    i32_ctx c = {out, seed, m ? m : 1};
    parallel_for(n, nthreads, fill_mod, &c, 65536);
}

void synth_i32_ascending(int32_t* out, size_t n, int nthreads) {
    i32_ctx c = {out, 0, 0};
    parallel_for(n, nthreads, fill_ascending, &c, 65536);
}

/* ---- float32 workloads -------------------------------------------------- */

typedef struct {
    float* out;
    uint64_t seed;
} f32_ctx;

/* Uniform double in (0, 1]: 53 random bits, shifted away from zero so that
 * log() below is finite. */
static inline double unit_open0(uint64_t x) {
    return ((double)(x >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}

static void fill_normal(void* p, size_t lo, size_t hi) {
    f32_ctx* c = (f32_ctx*)p;
    const double two_pi = 6.283185307179586476925286766559;
    for (size_t e = lo; e < hi; ++e) {
        size_t pair = e >> 1;
        double u1 = unit_open0(synth_splitmix64_at(c->seed, 2 * pair));
        double u2 = unit_open0(synth_splitmix64_at(c->seed, 2 * pair + 1));
        double r = sqrt(-2.0 * log(u1));
        double z = (e & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
        c->out[e] = (float)z;
    }
}

void synth_f32_normal(float* out, size_t n, uint64_t seed, int nthreads) {
    f32_ctx c = {out, seed};
    parallel_for(n, nthreads, fill_normal, &c, 65536);
}

typedef struct {
    float* x;
    int cols;
    int m;
    uint64_t seed;
} ties_ctx;

static void force_ties_rows(void* p, size_t lo, size_t hi) {
    ties_ctx* c = (ties_ctx*)p;
    int cols = c->cols;
    int* perm = (int*)malloc(sizeof(int) * (size_t)cols);
    if (!perm) return;
    for (size_t r = lo; r < hi; ++r) {
        float* row = c->x + r * (size_t)cols;
        float mx = row[0];
        for (int j = 1; j < cols; ++j)
            if (row[j] > mx) mx = row[j];
        uint64_t rs = synth_splitmix64_at(c->seed ^ ROW_STREAM_SALT, r);
        for (int j = 0; j < cols; ++j) perm[j] = j;
        for (int j = 0; j < c->m && j < cols; ++j) {
            uint64_t span = (uint64_t)(cols - j);
            int pick = j + (int)(synth_splitmix64_at(rs, (uint64_t)j) % span);
            int tmp = perm[j];
            perm[j] = perm[pick];
            perm[pick] = tmp;
            row[perm[j]] = mx;
        }
    }
    free(perm);
}

/* Overwrite m distinct positions of every row with that row's maximum. */
void synth_f32_force_ties(float* x, int rows, int cols, int m, uint64_t seed, int nthreads) {
    if (rows <= 0 || cols <= 0) return;
    ties_ctx c = {x, cols, m, seed};
    parallel_for((size_t)rows, nthreads, force_ties_rows, &c, 8);
}
