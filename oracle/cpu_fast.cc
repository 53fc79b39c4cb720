// The fast CPU baseline for int32 TopK -- NOT the oracle, and not used to
// check anything.  bench.py times it next to the oracle so that the GPU
// figure has a multi-core CPU figure beside the single-core one the TopK
// page reports ("CUDA parallel optimisation: TopK, shared memory and
// two-stage reduction", section 4.1, CPU column).
//
// The same two-stage shape as the GPU method, on host threads: every thread
// takes one contiguous chunk, keeps its k largest with std::nth_element,
// and one final std::nth_element + std::sort over the threads' candidates
// gives the answer.
#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <functional>
#include <thread>
#include <vector>

extern "C" {

// Threads the machine offers (std::thread::hardware_concurrency, at least 1).
int cpu_fast_hardware_threads(void) {
    const unsigned h = std::thread::hardware_concurrency();
    return h == 0 ? 1 : (int)h;
}

// The k largest of in[0..n), sorted descending, into out[0..k), with
// `threads` host threads (<= 0: all of them).  Returns the number of threads
// used, or -1 for bad arguments.
int cpu_fast_topk_i32(const int32_t* in, size_t n, int k, int32_t* out, int threads) {
    if (!in || !out || n == 0 || k < 1 || (size_t)k > n) return -1;
    int t = threads > 0 ? threads : cpu_fast_hardware_threads();
    const size_t kk = (size_t)k;
    // Every chunk must hold at least k elements.
    if ((size_t)t > n / kk) t = (int)std::max<size_t>(1, n / kk);
    std::vector<std::vector<int32_t>> part(t);
    std::vector<std::thread> pool;
    const size_t chunk = (n + (size_t)t - 1) / (size_t)t;
    for (int i = 0; i < t; ++i) {
        pool.emplace_back([&, i] {
            const size_t lo = std::min(n, (size_t)i * chunk), hi = std::min(n, lo + chunk);
            std::vector<int32_t>& v = part[i];
            v.assign(in + lo, in + hi);
            if (v.size() > kk) {
                std::nth_element(v.begin(), v.begin() + (kk - 1), v.end(), std::greater<int32_t>());
                v.resize(kk);
            }
        });
    }
    for (auto& th : pool) th.join();
    std::vector<int32_t> all;
    for (auto& v : part) all.insert(all.end(), v.begin(), v.end());
    std::nth_element(all.begin(), all.begin() + (kk - 1), all.end(), std::greater<int32_t>());
    std::sort(all.begin(), all.begin() + kk, std::greater<int32_t>());
    std::copy(all.begin(), all.begin() + kk, out);
    return t;
}

}  // extern "C"
