// Bucketed reduce-scatter of N_d 16-bit gradient replicas into fp32 shards.
//
// "第 5 课：ZeRO 与 FSDP" §3 step 1: each rank receives and sums only its 1/N_d
// slice of the gradients; "ZeRO: Memory Optimizations Toward Training Trillion
// Parameter Models" reading notes §4.1-§4.2: one reduce-scatter per bucket as
// backward fills it; §2.2: the fused buffers are kept in fp32.
//
// On one GPU the N_d ranks are N_d buffers, so the collective is a streaming
// kernel: one 32-byte load per rank per 16 elements, a binary32 sum in rank
// order, an IEEE division by N_d * loss_scale, 32-byte stores into the
// owner's fp32 shard, and the 32-element sums of squares for the global norm.
#include "zero_launch.h"

namespace zk {

template <int ND, class F>
__device__ __forceinline__ void rs_body(const RsArgs& a) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t gw = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    const uint32_t nw = (gridDim.x * kThreads) >> 5;
    const int nd = ND > 0 ? ND : a.nd;
    const float D = __fmul_rn((float)nd, a.st->loss_scale);
    bool bad = false;
    for (uint32_t base = a.seg.v_begin + gw * 32u; base < a.seg.v_end; base += nw * 32u) {
        const uint32_t v = base + lane;
        const bool active = v < a.seg.v_end;
        float g[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) g[e] = 0.0f;
        if (active) {
            float s[8];
            reduce8<ND, F>(a.rep, nd, v, a.seg.real_end, s);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                bad |= !isfinite(s[e]);
                g[e] = __fdiv_rn(s[e], D);
            }
            const uint32_t k = v - a.seg.seg_v;
            const uint32_t r = k / a.seg.shard_v;
            const uint32_t j = a.seg.base_v + (k - r * a.seg.shard_v);
            st8(a.gshard[r] + (size_t)j * kVec, g);
        }
        const float part = group32_sumsq(g);
        if (active && (lane & 3u) == 0u) a.partials[v >> 2] = part;
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0u) atomicOr(&a.st->nonfinite, 1);
}

template <int ND, class F>
__global__ void __launch_bounds__(kThreads) rs_kernel(const __grid_constant__ RsArgs a) {
    rs_body<ND, F>(a);
}

// 16 elements per thread (32-byte loads per rank): two lanes own one 32-element
// norm group.  Compile-time ND only.
template <int ND, class F>
__global__ void __launch_bounds__(kThreads) rs16_kernel(const __grid_constant__ RsArgs a) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t gw = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    const uint32_t nw = (gridDim.x * kThreads) >> 5;
    const float D = __fmul_rn((float)ND, a.st->loss_scale);
    const uint32_t vb = a.seg.v_begin >> 1, ve = a.seg.v_end >> 1;  // 16-element vectors
    const uint32_t seg16 = a.seg.seg_v >> 1, sh16 = a.seg.shard_v >> 1, base16 = a.seg.base_v >> 1;
    bool bad = false;
    for (uint32_t base = vb + gw * 32u; base < ve; base += nw * 32u) {
        const uint32_t v = base + lane;
        const bool active = v < ve;
        float g[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) g[e] = 0.0f;
        if (active) {
            float s[16];
            reduce16<ND, F>(a.rep, v, a.seg.real_end, s);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                bad |= !isfinite(s[e]);
                g[e] = __fdiv_rn(s[e], D);
            }
            const uint32_t k = v - seg16;
            const uint32_t r = k / sh16;
            const uint32_t j = base16 + (k - r * sh16);
            float* dst = a.gshard[r] + (size_t)j * 16;
            st8(dst, *reinterpret_cast<const float(*)[8]>(&g[0]));
            st8(dst + 8, *reinterpret_cast<const float(*)[8]>(&g[8]));
        }
        float hi = 0.0f, lo = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc_sq(g[e], hi, lo);
        combine_lanes(hi, lo, 1);
        if (active && (lane & 1u) == 0u) a.partials[v >> 1] = __fadd_rn(hi, lo);
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0u) atomicOr(&a.st->nonfinite, 1);
}

}  // namespace zk

using namespace zero_detail;

template <class K>
static zero_status_t launch_rs_kernel(K kern, const zk::RsArgs& a, int64_t nvec, cudaStream_t s) {
    kern<<<persistent_grid(kern, (nvec + zk::kThreads - 1) / zk::kThreads), zk::kThreads, 0, s>>>(a);
    return after_launch("zero_reduce_scatter");
}

// Compile-time rank counts take the 16-element kernel (32-byte loads; 6.98
// TB/s on the 1.5B buckets against 6.43 TB/s for 16-byte loads); other rank
// counts the 8-element kernel with a runtime rank loop.
template <int ND, class F>
static zero_status_t launch_rs(const zk::RsArgs& a, int64_t nvec, cudaStream_t s) {
    if constexpr (ND > 0) return launch_rs_kernel(zk::rs16_kernel<ND, F>, a, nvec / 2, s);
    return launch_rs_kernel(zk::rs_kernel<ND, F>, a, nvec, s);
}

extern "C" zero_status_t zero_reduce_scatter(const zero_layout* L, int32_t bucket_or_unit,
                                             const void* const* grad_replicas,
                                             float* const* grad_shards, zero_step_state* st,
                                             void* workspace, zero_stream_t stream) {
    clear_error();
    if (!L) return fail(ZERO_ERR_INVALID, "zero_reduce_scatter: NULL layout");
    if (L->stage == 0) return fail(ZERO_ERR_STATE, "zero_reduce_scatter: stage 0 has no partitioned step");
    if (bucket_or_unit < 0 || bucket_or_unit >= (int32_t)L->buckets.size())
        return fail(ZERO_ERR_INVALID, "zero_reduce_scatter: bucket index out of range");
    zero_status_t rc;
    if ((rc = check_ptr_array(grad_replicas, L->n_d, "zero_reduce_scatter grad_replicas")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)grad_shards, L->n_d, "zero_reduce_scatter grad_shards")) != ZERO_OK)
        return rc;
    if ((rc = check_dev_ptr(st, "zero_reduce_scatter state")) != ZERO_OK) return rc;
    if ((rc = check_dev_ptr(workspace, "zero_reduce_scatter workspace")) != ZERO_OK) return rc;

    zk::RsArgs a{};
    for (int r = 0; r < L->n_d; ++r) {
        a.rep[r] = static_cast<const uint16_t*>(grad_replicas[r]);
        a.gshard[r] = grad_shards[r];
    }
    a.partials = static_cast<float*>(workspace);
    a.st = st;
    a.nd = L->n_d;
    const auto& bk = L->buckets[bucket_or_unit];
    a.seg = seg_args(L->segs[L->bucket_seg[bucket_or_unit]], bk.first, bk.second);
    const int64_t nvec = (bk.second - bk.first) / zk::kVec;
    if (nvec == 0) return ZERO_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int nd = L->n_d;
    ZK_DISPATCH(nd, L->dtype, return launch_rs<ND, F>(a, nvec, s));
    return ZERO_OK;
}
