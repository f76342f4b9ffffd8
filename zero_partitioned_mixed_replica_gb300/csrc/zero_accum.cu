// ZeRO-1 gradient accumulation over micro-batches: every rank keeps a full
// fp32 accumulator and adds each micro-batch's 16-bit gradient locally, with
// no communication ("ZeRO: Memory Optimizations Toward Training Trillion
// Parameter Models" reading notes §4.1: with P_os gradient accumulation
// needs no extra communication); after the last micro-batch one
// reduce-scatter of the fp32 accumulators produces the averaged gradient.
// "第 5 课：ZeRO 与 FSDP" §2 counts the 4 Psi per rank this costs.
#include "zero_launch.h"

namespace zk {

// acc_r = x_r (first micro-batch) or acc_r + x_r for every rank and element.
template <class F, bool FIRST>
__global__ void __launch_bounds__(kThreads) accum_kernel(const __grid_constant__ AccumArgs a) {
    const uint64_t total = (uint64_t)a.v_per_rank * (uint64_t)a.nd;
    for (uint64_t t = (uint64_t)blockIdx.x * kThreads + threadIdx.x; t < total;
         t += (uint64_t)gridDim.x * kThreads) {
        const uint32_t r = (uint32_t)(t / a.v_per_rank);
        const uint32_t v = (uint32_t)(t - (uint64_t)r * a.v_per_rank);
        const int64_t i0 = (int64_t)v * kVec;
        if (!(in_bounds(r + 1, a.bnd.nd) && in_bounds((uint64_t)i0 + kVec, a.bnd.rep))) continue;
        float x[8];
        if (i0 + kVec <= a.real_end) {
            unpack8<F>(ld_stream(a.rep[r] + i0), x);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = (i0 + e < a.real_end) ? F::dec1(a.rep[r][i0 + e]) : 0.0f;
        }
        float* acc = a.acc[r] + i0;
        if constexpr (!FIRST) {
            float o[8];
            ld8(acc, o);
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = __fadd_rn(o[e], x[e]);
        }
        st8(acc, x);
    }
}

// Reduce-scatter of fp32 accumulators: s = A_0 + A_1 + ... in rank order,
// g = s / (N_d * n_micro * loss_scale) into the owner's shard, norm partials
// per 32 elements, non-finite flag.
template <int ND>
__global__ void __launch_bounds__(kThreads) rs_acc_kernel(const __grid_constant__ RsAccArgs a) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t gw = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    const uint32_t nw = (gridDim.x * kThreads) >> 5;
    const int nd = ND > 0 ? ND : a.nd;
    const float D = __double2float_rn(__dmul_rn(__dmul_rn((double)nd, (double)a.n_micro), (double)a.st->loss_scale));
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
            const size_t i0 = (size_t)v * kVec;
            float s[8];
            ld8(a.acc[0] + i0, s);
            for (int r = 1; r < nd; ++r) {
                float t[8];
                ld8(a.acc[r] + i0, t);
#pragma unroll
                for (int e = 0; e < 8; ++e) s[e] = __fadd_rn(s[e], t[e]);
            }
            if ((int64_t)i0 + kVec > a.seg.real_end) {  // padding reads as 0
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if ((int64_t)i0 + e >= a.seg.real_end) s[e] = 0.0f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                bad |= !isfinite(s[e]);
                g[e] = div_rn(s[e], D);
            }
            st8(a.gshard[r] + (size_t)j * kVec, g);
        }
        const float part = group32_sumsq(g);
        if (active && (lane & 3u) == 0u && in_bounds((v >> 2) + 1, a.bnd.part)) a.partials[v >> 2] = part;
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0u) atomicOr(&a.st->nonfinite, 1);
}

}  // namespace zk

using namespace zero_detail;

extern "C" zero_status_t zero_accumulate_grads(const zero_layout* L, int32_t micro, const void* const* grad_replicas,
                                               float* const* acc_replicas, zero_stream_t stream) {
    clear_error();
    if (!L) return fail(ZERO_ERR_INVALID, "zero_accumulate_grads: NULL layout");
    if (L->stage != 1) return fail(ZERO_ERR_STATE, "zero_accumulate_grads: ZeRO-1 only (ZeRO-2/3 reduce every micro-batch)");
    if (micro < 0) return fail(ZERO_ERR_INVALID, "zero_accumulate_grads: micro must be >= 0");
    zero_status_t rc;
    if ((rc = check_ptr_array(grad_replicas, L->n_d, "zero_accumulate_grads grad_replicas")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)acc_replicas, L->n_d, "zero_accumulate_grads acc")) != ZERO_OK)
        return rc;
    zk::AccumArgs a{};
    for (int r = 0; r < L->n_d; ++r) {
        a.rep[r] = static_cast<const uint16_t*>(grad_replicas[r]);
        a.acc[r] = acc_replicas[r];
    }
    a.v_per_rank = (uint32_t)(L->psi_pad / zk::kVec);
    a.real_end = L->segs[0].offset + L->segs[0].real;
    a.nd = L->n_d;
    a.bnd = make_bounds(L, 0);
    const int64_t work = ((int64_t)a.v_per_rank * a.nd + zk::kThreads - 1) / zk::kThreads;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (L->dtype == ZERO_BF16) {
        if (micro == 0) { auto k = zk::accum_kernel<zk::Bf16, true>; k<<<persistent_grid(k, work), zk::kThreads, 0, s>>>(a); }
        else { auto k = zk::accum_kernel<zk::Bf16, false>; k<<<persistent_grid(k, work), zk::kThreads, 0, s>>>(a); }
    } else {
        if (micro == 0) { auto k = zk::accum_kernel<zk::Fp16, true>; k<<<persistent_grid(k, work), zk::kThreads, 0, s>>>(a); }
        else { auto k = zk::accum_kernel<zk::Fp16, false>; k<<<persistent_grid(k, work), zk::kThreads, 0, s>>>(a); }
    }
    return after_launch("zero_accumulate_grads");
}

template <int ND>
static zero_status_t launch_rs_acc(const zk::RsAccArgs& a, int64_t nvec, cudaStream_t s) {
    auto k = zk::rs_acc_kernel<ND>;
    k<<<persistent_grid(k, (nvec + zk::kThreads - 1) / zk::kThreads), zk::kThreads, 0, s>>>(a);
    return after_launch("zero_reduce_scatter_accumulated");
}

extern "C" zero_status_t zero_reduce_scatter_accumulated(const zero_layout* L, int32_t bucket,
                                                         const float* const* acc_replicas, float* const* grad_shards,
                                                         int32_t n_micro, zero_step_state* st, void* workspace,
                                                         zero_stream_t stream) {
    clear_error();
    if (!L) return fail(ZERO_ERR_INVALID, "zero_reduce_scatter_accumulated: NULL layout");
    if (L->stage != 1) return fail(ZERO_ERR_STATE, "zero_reduce_scatter_accumulated: ZeRO-1 only");
    if (bucket < 0 || bucket >= (int32_t)L->buckets.size())
        return fail(ZERO_ERR_INVALID, "zero_reduce_scatter_accumulated: bucket index out of range");
    if (n_micro < 1) return fail(ZERO_ERR_INVALID, "zero_reduce_scatter_accumulated: n_micro must be >= 1");
    zero_status_t rc;
    const char* what = "zero_reduce_scatter_accumulated";
    if ((rc = check_ptr_array((const void* const*)acc_replicas, L->n_d, what)) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)grad_shards, L->n_d, what)) != ZERO_OK) return rc;
    if ((rc = check_dev_ptr(st, what)) != ZERO_OK) return rc;
    if ((rc = check_dev_ptr(workspace, what)) != ZERO_OK) return rc;
    zk::RsAccArgs a{};
    for (int r = 0; r < L->n_d; ++r) {
        a.acc[r] = acc_replicas[r];
        a.gshard[r] = grad_shards[r];
    }
    a.partials = static_cast<float*>(workspace);
    a.st = st;
    a.nd = L->n_d;
    a.n_micro = n_micro;
    a.bnd = make_bounds(L, 0);
    const auto& bk = L->buckets[bucket];
    a.seg = seg_args(L->segs[L->bucket_seg[bucket]], bk.first, bk.second);
    const int64_t nvec = (bk.second - bk.first) / zk::kVec;
    if (nvec == 0) return ZERO_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (L->n_d) {
        case 1: return launch_rs_acc<1>(a, nvec, s);
        case 2: return launch_rs_acc<2>(a, nvec, s);
        case 4: return launch_rs_acc<4>(a, nvec, s);
        case 8: return launch_rs_acc<8>(a, nvec, s);
        default: return launch_rs_acc<0>(a, nvec, s);
    }
}
