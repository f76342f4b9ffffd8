// All-gather of 16-bit parameter shards: the unfused ZeRO-1/2 all-gather
// ("第 5 课：ZeRO 与 FSDP" §3 step 3) and the ZeRO-3 per-unit gather into a
// transient buffer before forward and again before backward ("第 5 课" Fig. 5-1;
// reading notes "ZeRO: Memory Optimizations Toward Training Trillion Parameter
// Models" §3.1 and §4.3; "ZeRO-3 核心流程" §2 steps 1-2).
//
// Destination element i comes from rank r = i / S_u at shard offset
// base + i - r*S_u; every source vector is read once and written to all N_d
// destinations.  The unit's padding is not written.
#include "zero_launch.h"

namespace zk {

template <int ND>
__global__ void __launch_bounds__(kThreads) gather_kernel(const __grid_constant__ GatherArgs a) {
    const int nd = ND > 0 ? ND : a.nd;
    const uint32_t nvec = (uint32_t)((a.n_elems + kVec - 1) / kVec);
    for (uint32_t v = blockIdx.x * kThreads + threadIdx.x; v < nvec; v += gridDim.x * kThreads) {
        const uint32_t r = v / a.shard_v;
        const size_t so = ((size_t)a.base_v + (v - r * a.shard_v)) * kVec;
        const int64_t i0 = (int64_t)v * kVec;
        const int64_t i1 = i0 + kVec <= a.n_elems ? i0 + kVec : a.n_elems;
        if (!(in_bounds(r + 1, a.bnd.nd) && in_bounds(so + (uint64_t)(i1 - i0), a.bnd.src) &&
              in_bounds((uint64_t)i1, a.bnd.out)))
            continue;
        if (i0 + kVec <= a.n_elems) {
            const uint4 x = ld_stream(a.src[r] + so);
            if constexpr (ND > 0) {
#pragma unroll
                for (int q = 0; q < ND; ++q) st_stream(a.dst[q] + i0, x);
            } else {
                for (int q = 0; q < nd; ++q) st_stream(a.dst[q] + i0, x);
            }
        } else {
            const int tail = (int)(a.n_elems - i0);
            for (int e = 0; e < tail; ++e) {
                const uint16_t x = a.src[r][so + e];
                for (int q = 0; q < nd; ++q) a.dst[q][i0 + e] = x;
            }
        }
    }
}

struct CastArgs {
    const float* master[kMaxRanks];
    uint16_t* out[kMaxRanks];
    Bounds bnd;
    uint32_t shard_v;  // per-rank shard length / 8
    uint32_t total_v;  // nd * shard_v
    int32_t nd;
};

// Round-to-nearest-even cast of every rank's fp32 master shard to 16 bits,
// written the way the update's epilogue writes it: ZeRO-1/2 full replicas
// receive rank r's shard at its flat position in every replica (cast +
// all-gather, "第 5 课" §3 steps 2-3); shard outputs receive it in the rank's
// own 16-bit shard (ZeRO-3).
template <int ND, class F, int OUT>
__global__ void __launch_bounds__(kThreads) cast_kernel(const __grid_constant__ CastArgs a) {
    const int nd = ND > 0 ? ND : a.nd;
    for (uint32_t v = blockIdx.x * kThreads + threadIdx.x; v < a.total_v; v += gridDim.x * kThreads) {
        const uint32_t r = v / a.shard_v;
        const size_t o = (size_t)(v - r * a.shard_v) * kVec;
        const uint64_t out_end = OUT == ZERO_OUT_FULL_REPLICAS ? (uint64_t)(v + 1) * kVec : o + kVec;
        if (!(in_bounds(r + 1, a.bnd.nd) && in_bounds(o + kVec, a.bnd.shard) && in_bounds(out_end, a.bnd.out)))
            continue;
        float p[8];
        ld8(a.master[r] + o, p);
        const uint4 h = pack8<F>(p);
        if constexpr (OUT == ZERO_OUT_FULL_REPLICAS) {
            const size_t fo = (size_t)v * kVec;  // ZeRO-1/2: rank-major shard order is flat order
            if constexpr (ND > 0) {
#pragma unroll
                for (int q = 0; q < ND; ++q) st_stream(a.out[q] + fo, h);
            } else {
                for (int q = 0; q < nd; ++q) st_stream(a.out[q] + fo, h);
            }
        } else {
            st_stream(a.out[r] + o, h);
        }
    }
}

}  // namespace zk

using namespace zero_detail;

template <int ND, class F>
static zero_status_t launch_cast(const zk::CastArgs& a, int32_t out_kind, cudaStream_t s) {
    const int64_t work = ((int64_t)a.total_v + zk::kThreads - 1) / zk::kThreads;
    if (out_kind == ZERO_OUT_FULL_REPLICAS) {
        auto kern = zk::cast_kernel<ND, F, ZERO_OUT_FULL_REPLICAS>;
        kern<<<persistent_grid(kern, work), zk::kThreads, 0, s>>>(a);
    } else {
        auto kern = zk::cast_kernel<ND, F, ZERO_OUT_SHARDS>;
        kern<<<persistent_grid(kern, work), zk::kThreads, 0, s>>>(a);
    }
    return after_launch("zero_cast_params");
}

extern "C" zero_status_t zero_cast_params(const zero_layout* L, const float* const* master,
                                          void* const* param16_out, int32_t out_kind, zero_stream_t stream) {
    clear_error();
    if (!L) return fail(ZERO_ERR_INVALID, "zero_cast_params: NULL layout");
    if (L->stage == 0) return fail(ZERO_ERR_STATE, "zero_cast_params: stage 0 has no partitioned state");
    if (out_kind != ZERO_OUT_FULL_REPLICAS && out_kind != ZERO_OUT_SHARDS)
        return fail(ZERO_ERR_INVALID, "zero_cast_params: unknown out_kind");
    if (L->stage == 3 && out_kind != ZERO_OUT_SHARDS)
        return fail(ZERO_ERR_STATE, "zero_cast_params: ZeRO-3 writes 16-bit shards only");
    zero_status_t rc;
    if ((rc = check_ptr_array((const void* const*)master, L->n_d, "zero_cast_params master")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)param16_out, L->n_d, "zero_cast_params param16_out")) != ZERO_OK)
        return rc;
    zk::CastArgs a{};
    for (int r = 0; r < L->n_d; ++r) {
        a.master[r] = master[r];
        a.out[r] = static_cast<uint16_t*>(param16_out[r]);
    }
    a.shard_v = (uint32_t)(L->shard_len / zk::kVec);
    a.total_v = (uint32_t)((int64_t)L->n_d * (L->shard_len / zk::kVec));
    a.nd = L->n_d;
    a.bnd = make_bounds(L, out_kind == ZERO_OUT_FULL_REPLICAS ? L->psi_pad : L->shard_len);
    if (a.total_v == 0) return ZERO_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ZK_DISPATCH(L->n_d, L->dtype, return launch_cast<ND, F>(a, out_kind, s));
    return ZERO_OK;
}

// Resident CTAs per SM: at N_d = 2, launches long enough to give every thread
// ~64 vectors at 6 CTAs per SM run faster with 6 than with all 8 that fit
// (7B block unit, 202M elements: 0.2024 -> 0.1971 ms on GB300); shorter ones
// (350M units of 12.6M elements: 0.909 -> 0.942 ms per step at 6) and other
// N_d (no difference measured) keep the full grid.
template <int ND>
static zero_status_t launch_gather(const zk::GatherArgs& a, const char* what, cudaStream_t s) {
    const int64_t nvec = (a.n_elems + zk::kVec - 1) / zk::kVec;
    auto kern = zk::gather_kernel<ND>;
    int64_t work = (nvec + zk::kThreads - 1) / zk::kThreads;
    const int64_t sms = sm_count() > 0 ? sm_count() : 1;
    if (a.nd == 2 && nvec >= 64 * 6 * sms * zk::kThreads && work > 6 * sms) work = 6 * sms;
    kern<<<persistent_grid(kern, work), zk::kThreads, 0, s>>>(a);
    return after_launch(what);
}

static zero_status_t dispatch_gather(int nd, const zk::GatherArgs& a, const char* what, cudaStream_t s) {
    if (a.n_elems == 0) return ZERO_OK;
    switch (nd) {
        case 1: return launch_gather<1>(a, what, s);
        case 2: return launch_gather<2>(a, what, s);
        case 4: return launch_gather<4>(a, what, s);
        case 8: return launch_gather<8>(a, what, s);
        default: return launch_gather<0>(a, what, s);
    }
}

extern "C" zero_status_t zero_allgather_params(const zero_layout* L, const void* const* param16_shards,
                                               void* const* param16_full, zero_stream_t stream) {
    clear_error();
    if (!L) return fail(ZERO_ERR_INVALID, "zero_allgather_params: NULL layout");
    if (L->stage == 0 || L->stage == 3)
        return fail(ZERO_ERR_STATE, "zero_allgather_params: ZeRO-1/2 only (ZeRO-3 gathers per unit)");
    zero_status_t rc;
    if ((rc = check_ptr_array(param16_shards, L->n_d, "zero_allgather_params shards")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)param16_full, L->n_d, "zero_allgather_params full")) != ZERO_OK)
        return rc;
    zk::GatherArgs a{};
    for (int r = 0; r < L->n_d; ++r) {
        a.src[r] = static_cast<const uint16_t*>(param16_shards[r]);
        a.dst[r] = static_cast<uint16_t*>(param16_full[r]);
    }
    const zero_segment& sg = L->segs[0];
    a.shard_v = (uint32_t)(sg.shard / zk::kVec);
    a.base_v = 0;
    a.n_elems = L->psi_pad;
    a.nd = L->n_d;
    a.bnd = make_bounds(L, L->psi_pad);
    return dispatch_gather(L->n_d, a, "zero_allgather_params", reinterpret_cast<cudaStream_t>(stream));
}

extern "C" zero_status_t zero_stage3_gather_layer(const zero_layout* L, int32_t unit,
                                                  const void* const* param16_shards, void* const* transient,
                                                  zero_stream_t stream) {
    clear_error();
    if (!L) return fail(ZERO_ERR_INVALID, "zero_stage3_gather_layer: NULL layout");
    if (L->stage != 3) return fail(ZERO_ERR_STATE, "zero_stage3_gather_layer: ZeRO-3 only");
    if (unit < 0 || unit >= (int32_t)L->segs.size())
        return fail(ZERO_ERR_INVALID, "zero_stage3_gather_layer: unit index out of range");
    zero_status_t rc;
    if ((rc = check_ptr_array(param16_shards, L->n_d, "zero_stage3_gather_layer shards")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)transient, L->n_d, "zero_stage3_gather_layer transient")) != ZERO_OK)
        return rc;
    zk::GatherArgs a{};
    for (int r = 0; r < L->n_d; ++r) {
        a.src[r] = static_cast<const uint16_t*>(param16_shards[r]);
        a.dst[r] = static_cast<uint16_t*>(transient[r]);
    }
    const zero_segment& sg = L->segs[unit];
    a.shard_v = (uint32_t)(sg.shard / zk::kVec);
    a.base_v = (uint32_t)(sg.shard_base / zk::kVec);
    a.n_elems = sg.real;
    a.nd = L->n_d;
    a.bnd = make_bounds(L, sg.real);   // a transient holds at least the unit's real size
    return dispatch_gather(L->n_d, a, "zero_stage3_gather_layer", reinterpret_cast<cudaStream_t>(stream));
}
