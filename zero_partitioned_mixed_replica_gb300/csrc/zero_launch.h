// Host-side launch helpers shared by libzero's CUDA translation units.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <unordered_map>
#include <string>

#include "zero_device.cuh"
#include "zero_internal.h"

namespace zero_detail {

inline int sm_count() {
    static std::atomic<int> cache[64];  // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Persistent grid: every CTA resident at once (SMs x resident CTAs per SM),
// capped by the CTAs the work needs; kernels grid-stride over the rest.
template <class Kernel>
inline int persistent_grid(Kernel kernel, int64_t work_ctas, size_t dyn_smem = 0, int threads = zk::kThreads) {
    // resident CTAs per SM, cached per (device, kernel address)
    static std::mutex mu;
    static std::unordered_map<const void*, int> cache[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache[dev].find(reinterpret_cast<const void*>(kernel));
        if (it != cache[dev].end()) per_sm = it->second;
    }
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, dyn_smem) != cudaSuccess ||
            per_sm <= 0)
            per_sm = 1;
        std::lock_guard<std::mutex> lock(mu);
        cache[dev][reinterpret_cast<const void*>(kernel)] = per_sm;
    }
    int sms = sm_count();
    if (sms <= 0) sms = 1;
    int64_t cap = (int64_t)sms * per_sm;
    const int32_t user_cap = max_ctas();
    if (user_cap > 0 && user_cap < cap) cap = user_cap;
    int64_t g = work_ctas < cap ? work_ctas : cap;
    return g < 1 ? 1 : (int)g;
}

inline zero_status_t check_dev_ptr(const void* p, const char* what) {
    if (!p) return fail(ZERO_ERR_INVALID, std::string(what) + ": NULL device pointer");
    if (reinterpret_cast<uintptr_t>(p) & 255u)
        return fail(ZERO_ERR_ALIGN, std::string(what) + ": device pointer not 256-byte aligned");
    return ZERO_OK;
}

inline zero_status_t check_ptr_array(const void* const* arr, int n, const char* what) {
    if (!arr) return fail(ZERO_ERR_INVALID, std::string(what) + ": NULL pointer array");
    for (int i = 0; i < n; ++i) {
        zero_status_t s = check_dev_ptr(arr[i], what);
        if (s != ZERO_OK) return s;
    }
    return ZERO_OK;
}

inline zero_status_t after_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(ZERO_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
    count_launches(1);
    return ZERO_OK;
}

// The extents a launch's accesses are checked against (bounds-checked
// builds; the normal build carries them unused): from the layout, each
// shortened by the test hook's slack.  out_elems: each 16-bit output's size.
inline zk::Bounds make_bounds(const zero_layout* L, int64_t out_elems) {
    const int64_t sl = check_slack();
    auto cut = [sl](int64_t x) { return (uint64_t)(x > sl ? x - sl : 0); };
    zk::Bounds b{};
    b.rep = cut(L->psi_pad);
    b.shard = cut(L->shard_len);
    b.out = cut(out_elems);
    b.part = cut(partials_count(L));
    b.src = cut(L->shard_len);
    b.nd = (uint32_t)L->n_d;
    return b;
}

inline zk::SegArgs seg_args(const zero_segment& s, int64_t begin, int64_t end) {
    zk::SegArgs a;
    a.v_begin = (uint32_t)(begin / zk::kVec);
    a.v_end = (uint32_t)(end / zk::kVec);
    a.seg_v = (uint32_t)(s.offset / zk::kVec);
    a.shard_v = (uint32_t)(s.shard / zk::kVec);
    a.base_v = (uint32_t)(s.shard_base / zk::kVec);
    a.pad0 = 0;
    a.real_end = s.offset + s.real;
    return a;
}

}  // namespace zero_detail

#ifdef ZK_CHECKED
// This translation unit's counter of skipped accesses, read through the
// registry (zero_bounds_violations).
namespace {
int zk_read_bounds_hits(int64_t* out, bool reset) {
    cudaError_t e = cudaDeviceSynchronize();
    unsigned long long v = 0;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, zk::zk_bounds_hits, sizeof v);
    if (e == cudaSuccess && reset) {
        const unsigned long long z = 0;
        e = cudaMemcpyToSymbol(zk::zk_bounds_hits, &z, sizeof z);
    }
    *out += (int64_t)v;
    return e == cudaSuccess ? 0 : 1;
}
const bool zk_bounds_registered = (zero_detail::register_bounds_reader(&zk_read_bounds_hits), true);
}  // namespace
#endif

#define ZK_ND_SWITCH(nd, ...)                                  \
    switch (nd) {                                              \
        case 1: { constexpr int ND = 1; __VA_ARGS__; } break;  \
        case 2: { constexpr int ND = 2; __VA_ARGS__; } break;  \
        case 4: { constexpr int ND = 4; __VA_ARGS__; } break;  \
        case 8: { constexpr int ND = 8; __VA_ARGS__; } break;  \
        default: { constexpr int ND = 0; __VA_ARGS__; } break; \
    }

#define ZK_DISPATCH(nd, dtype, ...)                                  \
    do {                                                             \
        if ((dtype) == ZERO_BF16) {                                  \
            using F = zk::Bf16;                                      \
            ZK_ND_SWITCH(nd, __VA_ARGS__)                            \
        } else {                                                     \
            using F = zk::Fp16;                                      \
            ZK_ND_SWITCH(nd, __VA_ARGS__)                            \
        }                                                            \
    } while (0)
