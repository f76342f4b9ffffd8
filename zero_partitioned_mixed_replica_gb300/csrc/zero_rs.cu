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

// D = binary32(N_d * n_micro * loss_scale): the exact product rounded once.
__device__ __forceinline__ float rs_divisor(int nd, int n_micro, float loss_scale) {
    return __double2float_rn(__dmul_rn(__dmul_rn((double)nd, (double)n_micro), (double)loss_scale));
}

// Combine the rank-order sum s with the accumulator for the reduce-scatter
// mode; returns the value stored (g, or the running accumulator).
template <int MODE>
__device__ __forceinline__ void rs_combine(float (&s)[8], const float* accp, float D, bool& bad) {
    if constexpr (MODE == RS_PLAIN) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            bad |= !isfinite(s[e]);
            s[e] = div_rn(s[e], D);
        }
    } else if constexpr (MODE == RS_FIRST) {
        (void)accp;
    } else {
        float acc[8];
        ld8(accp, acc);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float t = __fadd_rn(acc[e], s[e]);
            if constexpr (MODE == RS_LAST) {
                bad |= !isfinite(t);
                s[e] = div_rn(t, D);
            } else {
                s[e] = t;
            }
        }
    }
}

template <int ND, class F, int MODE>
__device__ __forceinline__ void rs_body(const RsArgs& a) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t gw = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    const uint32_t nw = (gridDim.x * kThreads) >> 5;
    const int nd = ND > 0 ? ND : a.nd;
    const float D = rs_divisor(nd, a.n_micro, a.st->loss_scale);
    bool bad = false;
    for (uint32_t base = a.seg.v_begin + gw * 32u; base < a.seg.v_end; base += nw * 32u) {
        const uint32_t v = base + lane;
        const bool active = v < a.seg.v_end;
        float g[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) g[e] = 0.0f;
        const uint32_t k = v - a.seg.seg_v;
        const uint32_t r = k / a.seg.shard_v;
        const uint32_t j = a.seg.base_v + (k - r * a.seg.shard_v);
        if (active && in_bounds((uint64_t)(v + 1) * kVec, a.bnd.rep) && in_bounds(r + 1, a.bnd.nd) &&
            in_bounds((uint64_t)(j + 1) * kVec, a.bnd.shard)) {
            float s[8];
            reduce8<ND, F>(a.rep, nd, v, a.seg.real_end, s);
            float* dst = a.gshard[r] + (size_t)j * kVec;
            rs_combine<MODE>(s, dst, D, bad);
#pragma unroll
            for (int e = 0; e < 8; ++e) g[e] = s[e];
            st8(dst, g);
        }
        if constexpr (MODE == RS_PLAIN || MODE == RS_LAST) {
            const float part = group32_sumsq(g);
            if (active && (lane & 3u) == 0u && in_bounds((v >> 2) + 1, a.bnd.part)) a.partials[v >> 2] = part;
        }
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0u) atomicOr(&a.st->nonfinite, 1);
}

template <int ND, class F, int MODE>
__global__ void __launch_bounds__(kThreads) rs_kernel(const __grid_constant__ RsArgs a) {
    rs_body<ND, F, MODE>(a);
}

// 16 elements per thread (32-byte loads per rank): two lanes own one 32-element
// norm group.  Compile-time ND only.
template <int ND, class F, int MODE>
__global__ void __launch_bounds__(kThreads) rs16_kernel(const __grid_constant__ RsArgs a) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t gw = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    const uint32_t nw = (gridDim.x * kThreads) >> 5;
    const float D = rs_divisor(ND, a.n_micro, a.st->loss_scale);
    const uint32_t vb = a.seg.v_begin >> 1, ve = a.seg.v_end >> 1;  // 16-element vectors
    const uint32_t seg16 = a.seg.seg_v >> 1, sh16 = a.seg.shard_v >> 1, base16 = a.seg.base_v >> 1;
    bool bad = false;
    for (uint32_t base = vb + gw * 32u; base < ve; base += nw * 32u) {
        const uint32_t v = base + lane;
        const bool active = v < ve;
        float g[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) g[e] = 0.0f;
        const uint32_t k = v - seg16;
        const uint32_t r = k / sh16;
        const uint32_t j = base16 + (k - r * sh16);
        if (active && in_bounds((uint64_t)(v + 1) * 16, a.bnd.rep) && in_bounds(r + 1, a.bnd.nd) &&
            in_bounds((uint64_t)(j + 1) * 16, a.bnd.shard)) {
            float s[16];
            reduce16<ND, F>(a.rep, v, a.seg.real_end, s);
            float* dst = a.gshard[r] + (size_t)j * 16;
            float* h0 = reinterpret_cast<float*>(&s[0]);
            rs_combine<MODE>(*reinterpret_cast<float(*)[8]>(h0), dst, D, bad);
            rs_combine<MODE>(*reinterpret_cast<float(*)[8]>(h0 + 8), dst + 8, D, bad);
#pragma unroll
            for (int e = 0; e < 16; ++e) g[e] = s[e];
            st8(dst, *reinterpret_cast<const float(*)[8]>(&g[0]));
            st8(dst + 8, *reinterpret_cast<const float(*)[8]>(&g[8]));
        }
        if constexpr (MODE == RS_PLAIN || MODE == RS_LAST) {
            float hi = 0.0f, lo = 0.0f;
#pragma unroll
            for (int e = 0; e < 16; ++e) acc_sq(g[e], hi, lo);
            combine_lanes(hi, lo, 1);
            if (active && (lane & 1u) == 0u && in_bounds((v >> 1) + 1, a.bnd.part))
                a.partials[v >> 1] = __fadd_rn(hi, lo);
        }
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
template <int ND, class F, int MODE>
static zero_status_t launch_rs_mode(const zk::RsArgs& a, int64_t nvec, cudaStream_t s) {
    if constexpr (ND > 0) return launch_rs_kernel(zk::rs16_kernel<ND, F, MODE>, a, nvec / 2, s);
    return launch_rs_kernel(zk::rs_kernel<ND, F, MODE>, a, nvec, s);
}

template <int ND, class F>
static zero_status_t launch_rs(const zk::RsArgs& a, int64_t nvec, int mode, cudaStream_t s) {
    switch (mode) {
        case zk::RS_FIRST: return launch_rs_mode<ND, F, zk::RS_FIRST>(a, nvec, s);
        case zk::RS_MIDDLE: return launch_rs_mode<ND, F, zk::RS_MIDDLE>(a, nvec, s);
        case zk::RS_LAST: return launch_rs_mode<ND, F, zk::RS_LAST>(a, nvec, s);
        default: return launch_rs_mode<ND, F, zk::RS_PLAIN>(a, nvec, s);
    }
}

static zero_status_t rs_common(const zero_layout* L, int32_t bucket_or_unit, const void* const* grad_replicas,
                               float* const* grad_shards, zero_step_state* st, void* workspace, int mode,
                               int32_t n_micro, zero_stream_t stream, const char* what) {
    zero_status_t rc;
    if ((rc = check_ptr_array(grad_replicas, L->n_d, what)) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)grad_shards, L->n_d, what)) != ZERO_OK) return rc;
    if ((rc = check_dev_ptr(st, what)) != ZERO_OK) return rc;
    if ((rc = check_dev_ptr(workspace, what)) != ZERO_OK) return rc;
    zk::RsArgs a{};
    for (int r = 0; r < L->n_d; ++r) {
        a.rep[r] = static_cast<const uint16_t*>(grad_replicas[r]);
        a.gshard[r] = grad_shards[r];
    }
    a.partials = static_cast<float*>(workspace);
    a.st = st;
    a.nd = L->n_d;
    a.n_micro = n_micro;
    a.bnd = make_bounds(L, 0);
    const auto& bk = L->buckets[bucket_or_unit];
    a.seg = seg_args(L->segs[L->bucket_seg[bucket_or_unit]], bk.first, bk.second);
    const int64_t nvec = (bk.second - bk.first) / zk::kVec;
    if (nvec == 0) return ZERO_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ZK_DISPATCH(L->n_d, L->dtype, return launch_rs<ND, F>(a, nvec, mode, s));
    return ZERO_OK;
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
    return rs_common(L, bucket_or_unit, grad_replicas, grad_shards, st, workspace, zk::RS_PLAIN, 1, stream,
                     "zero_reduce_scatter");
}

extern "C" zero_status_t zero_reduce_scatter_micro(const zero_layout* L, int32_t bucket_or_unit, int32_t micro,
                                                   int32_t n_micro, const void* const* grad_replicas,
                                                   float* const* acc_shards, zero_step_state* st, void* workspace,
                                                   zero_stream_t stream) {
    clear_error();
    if (!L) return fail(ZERO_ERR_INVALID, "zero_reduce_scatter_micro: NULL layout");
    if (L->stage != 2 && L->stage != 3)
        return fail(ZERO_ERR_STATE, "zero_reduce_scatter_micro: ZeRO-2/3 only (ZeRO-1 accumulates locally)");
    if (bucket_or_unit < 0 || bucket_or_unit >= (int32_t)L->buckets.size())
        return fail(ZERO_ERR_INVALID, "zero_reduce_scatter_micro: bucket index out of range");
    if (n_micro < 1 || micro < 0 || micro >= n_micro)
        return fail(ZERO_ERR_INVALID, "zero_reduce_scatter_micro: need 0 <= micro < n_micro");
    const int mode = n_micro == 1 ? zk::RS_PLAIN
                                  : (micro == 0 ? zk::RS_FIRST : (micro == n_micro - 1 ? zk::RS_LAST : zk::RS_MIDDLE));
    return rs_common(L, bucket_or_unit, grad_replicas, acc_shards, st, workspace, mode, n_micro, stream,
                     "zero_reduce_scatter_micro");
}
