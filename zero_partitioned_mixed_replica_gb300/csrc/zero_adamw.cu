// Sharded AdamW + cast to 16 bits + (fused) all-gather.
//
// "第 5 课：ZeRO 与 FSDP" §3 step 2: each rank updates its 1/N_d of the fp32
// master weights and optimizer state and casts the result to BF16 in place;
// step 3: an all-gather rebuilds every rank's full 16-bit parameters.  "ZeRO-3
// 核心流程" §2 step 3: the update is local, with zero communication.  The
// pages name AdamW (mixed precision, k = 12: fp32 master, m, v; reading notes
// §2.1) but give no formula; the update below is decoupled weight decay with
// bias corrections, one binary32 rounding per operation.
//
// With the N_d ranks as N_d buffers on one GPU, the all-gather becomes N_d
// bulk stores of the freshly cast tile from shared memory: the parameters
// never make a second trip through HBM.
#include "zero_launch.h"

namespace zk {

// A persistent CTA walks tiles of TE elements of the rank shards.  One thread
// issues 1-D bulk copies of g, p, m, v into a STAGES-deep shared-memory ring
// (completion counted on one mbarrier per stage); all warps update from
// shared memory into a double-buffered output stage; one thread then issues
// bulk stores of p, m, v and of the cast tile to every replica (or to the
// rank's 16-bit shard).  Global traffic leaves the load/store queues of the
// SMs entirely and moves in 4-8 KB transfers.
template <int TE, int STAGES, int OST>
struct AdamTmaSmem {
    static constexpr int kOst = OST;
    static constexpr size_t in_bytes = (size_t)STAGES * 4 * TE * sizeof(float);
    static constexpr size_t out_bytes = (size_t)kOst * 3 * TE * sizeof(float);
    static constexpr size_t h_bytes = (size_t)kOst * TE * sizeof(uint16_t);
    static constexpr size_t bar_off = in_bytes + out_bytes + h_bytes;
    static constexpr size_t total = bar_off + (size_t)STAGES * sizeof(uint64_t);
};

template <int ND, class F, int OUT, int TE, int STAGES, int OSTAGES, int NT>
__global__ void __launch_bounds__(NT, 1) adamw_tma_kernel(const __grid_constant__ AdamArgs a) {
    using SM = AdamTmaSmem<TE, STAGES, OSTAGES>;
    constexpr int OST = SM::kOst;
    constexpr int PARTS = TE / (NT * 4);  // float4 groups per thread per tile
    static_assert(PARTS >= 1 && TE % (NT * 4) == 0, "tile must give every thread whole float4 groups");
    extern __shared__ __align__(1024) unsigned char smem[];
    float* in = reinterpret_cast<float*>(smem);
    float* ob = reinterpret_cast<float*>(smem + SM::in_bytes);
    uint16_t* hb = reinterpret_cast<uint16_t*>(smem + SM::in_bytes + SM::out_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::bar_off);
    __shared__ AdamConsts sk;
    __shared__ int s_apply, s_abort;
    __shared__ uint32_t s_stop;
    const int tid = threadIdx.x;
    if (tid == 0) {
        const zero_step_state* st = a.st;
        s_apply = st->apply;
        s_abort = 0;
        sk = make_consts(st->beta1, st->beta2, st->beta1_pow, st->beta2_pow, a.lr, a.eps, a.wd,
                         st->clip_coef);
        for (int i = 0; i < STAGES; ++i) mbar_init(&full[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (!s_apply) return;  // overflow: the step is skipped
    const AdamConsts k = sk;
    const int nd = ND > 0 ? ND : a.nd;
    const uint64_t S = (uint64_t)a.shard_v * kVec;
    const uint32_t ntile = (uint32_t)((S + TE - 1) / TE);
    const uint32_t total = ntile * (uint32_t)nd;
    // Tiles are dealt to the CTAs round-robin: CTA c takes tiles c, c + G,
    // c + 2G, ...  An element whose gradient and moments are all zero (an
    // embedding row no batch has touched yet) sends both divisions of the
    // update down their slow path and costs about twice a dense one; dealt this
    // way a contiguous zero region spreads over every CTA.  GB300, 1.5B launch:
    // one contiguous range of tiles per CTA took 10.68 ms dense but 20.91 ms
    // with the word-embedding gradients zero (the few CTAs holding the zero
    // region set the time), round-robin 10.73 / 11.27 ms.  On the current
    // refill schedule, single tiles against batches of 4 consecutive tiles
    // round-robin: 10.716 / 10.750 and 10.726 / 10.762 ms (two boxes); batches
    // of 2 or 8: 10.820, 10.790.
    const uint32_t G = gridDim.x, c = blockIdx.x;
    const uint32_t count = c < total ? (total - c + G - 1) / G : 0u;

    // A tile whose extents fail the checked build's bounds test is processed
    // as empty (len 0): nothing is loaded or stored for it.
    auto tile_of = [&](uint32_t kk, uint32_t& r, uint64_t& j0, uint32_t& len) {
        const uint32_t T = c + kk * G;
        r = T / ntile;
        j0 = (uint64_t)(T - r * ntile) * TE;
        const uint64_t rem = S - j0;
        len = rem < (uint64_t)TE ? (uint32_t)rem : (uint32_t)TE;
        const uint64_t out_end = OUT == ZERO_OUT_FULL_REPLICAS ? (uint64_t)r * S + j0 + len : j0 + len;
        if (!(in_bounds(r + 1, a.bnd.nd) && in_bounds(j0 + len, a.bnd.shard) && in_bounds(out_end, a.bnd.out)))
            len = 0;
    };
    auto issue = [&](uint32_t kk) {  // one thread
        uint32_t r, len;
        uint64_t j0;
        tile_of(kk, r, j0, len);
        const int slot = (int)(kk % STAGES);
        float* dst = in + (size_t)slot * 4 * TE;
        const uint32_t bytes = len * (uint32_t)sizeof(float);
        mbar_arrive_expect_tx(&full[slot], 4u * bytes);
        if (kChecked && len == 0) return;
        bulk_g2s(dst, a.gshard[r] + j0, bytes, &full[slot]);
        bulk_g2s(dst + TE, a.master[r] + j0, bytes, &full[slot]);
        bulk_g2s(dst + 2 * TE, a.m[r] + j0, bytes, &full[slot]);
        bulk_g2s(dst + 3 * TE, a.v[r] + j0, bytes, &full[slot]);
    };
    // STAGES tiles in flight from the start; each tile's slot is refilled
    // (tile kk + STAGES) right after the tile's stores are issued, when every
    // thread has read it.  GB300, 1.5B launch: 10.647 ms against 10.673 ms
    // refilling at the top of the next iteration (STAGES - 1 tiles ahead).
    if (tid == 0)
        for (uint32_t kk = 0; kk < (uint32_t)STAGES && kk < count; ++kk) issue(kk);
    for (uint32_t kk = 0; kk < count; ++kk) {
        if (tid == 0) bulk_wait_read<OST - 1>();  // stores issued from output stage kk % OST have read it
        __syncthreads();
        const int slot = (int)(kk % STAGES);
        const int o = (int)(kk % OST);
        const bool ok = mbar_wait_bounded(&full[slot], (kk / STAGES) & 1u);
        if (!ok) {
            s_abort = 1;
            s_stop = kk;  // every thread that gives up writes the same tile index
            atomicOr(&a.st->error, ZERO_DEVERR_WAIT_TIMEOUT);
        }
        uint32_t r, len;
        uint64_t j0;
        tile_of(kk, r, j0, len);
        const float* src = in + (size_t)slot * 4 * TE;
        float* dst = ob + (size_t)o * 3 * TE;
        uint16_t* hd = hb + (size_t)o * TE;
        if (ok) {
#pragma unroll
            for (int part = 0; part < PARTS; ++part) {
                const int e = part * NT * 4 + tid * 4;
                if ((uint32_t)e < len) {
                    const float4 g4 = *reinterpret_cast<const float4*>(src + e);
                    float4 p4 = *reinterpret_cast<const float4*>(src + TE + e);
                    float4 m4 = *reinterpret_cast<const float4*>(src + 2 * TE + e);
                    float4 v4 = *reinterpret_cast<const float4*>(src + 3 * TE + e);
                    // the plain update: a zero-state test here (as in the other update
                    // kernels) evens out zero regions but cost 4% on dense gradients
                    // (1.5B launch 11.12 against 10.68 ms)
                    adamw1(p4.x, m4.x, v4.x, g4.x, k);
                    adamw1(p4.y, m4.y, v4.y, g4.y, k);
                    adamw1(p4.z, m4.z, v4.z, g4.z, k);
                    adamw1(p4.w, m4.w, v4.w, g4.w, k);
                    *reinterpret_cast<float4*>(dst + e) = p4;
                    *reinterpret_cast<float4*>(dst + TE + e) = m4;
                    *reinterpret_cast<float4*>(dst + 2 * TE + e) = v4;
                    uint2 h;
                    h.x = F::pack(p4.x, p4.y);
                    h.y = F::pack(p4.z, p4.w);
                    *reinterpret_cast<uint2*>(hd + e) = h;
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (s_abort) break;
        if (tid == 0 && (!kChecked || len != 0)) {
            const uint32_t fb = len * (uint32_t)sizeof(float);
            const uint32_t hbytes = len * (uint32_t)sizeof(uint16_t);
            bulk_s2g(a.master[r] + j0, dst, fb);
            bulk_s2g(a.m[r] + j0, dst + TE, fb);
            bulk_s2g(a.v[r] + j0, dst + 2 * TE, fb);
            if constexpr (OUT == ZERO_OUT_FULL_REPLICAS) {
                const uint64_t fo = (uint64_t)r * S + j0;  // ZeRO-1/2: rank-major order is flat order
                for (int q = 0; q < nd; ++q) bulk_s2g(a.out[q] + fo, hd, hbytes);
            } else {
                bulk_s2g(a.out[r] + j0, hd, hbytes);
            }
            bulk_commit();
        }
        if (tid == 0 && kk + STAGES < count) issue(kk + STAGES);  // into the slot tile kk released
    }
    if (tid == 0) {
        if (s_abort) {
            // After a timed-out wait on tile s_stop, let the loads still in
            // flight (tiles s_stop .. s_stop + STAGES - 1) land before the CTA
            // gives up its shared memory: up to kDrainTries bounded waits per
            // tile.  A tile that still has not landed is reported with
            // ZERO_DEVERR_DRAIN_TIMEOUT; the CTA then exits with that copy
            // possibly outstanding.
            const uint32_t k0 = s_stop, k1 = min(count, k0 + (uint32_t)STAGES);
            for (uint32_t j = k0; j < k1; ++j) {
                bool landed = false;
                for (int tries = 0; tries < kDrainTries && !landed; ++tries)
                    landed = mbar_wait_bounded(&full[j % STAGES], (j / STAGES) & 1u);
                if (!landed) atomicOr(&a.st->error, ZERO_DEVERR_DRAIN_TIMEOUT);
            }
        }
        bulk_wait_all<0>();
    }
}

// Four CTAs of 256 threads per SM (64 registers, no spills): the shard-output
// variant otherwise takes 68 registers and three CTAs, and at N_d = 2 its
// ~30 B/param leave it bound by latency (7B ZeRO-3 unit update 0.977 ->
// 0.941 ms).  Five CTAs per SM force spills.
// The same update with plain 32-byte loads and stores, 8 elements per thread
// over the rank-major shard space.  With few bytes per element (the 16-bit
// shard output of ZeRO-3) the TMA pipeline's per-tile barriers dominate and
// this form is faster; results are identical (same per-element update).
template <int ND, class F, int OUT>
__global__ void __launch_bounds__(kThreads, 4) adamw_ldg_kernel(const __grid_constant__ AdamArgs a) {
    __shared__ AdamConsts sk;
    __shared__ int s_apply;
    if (threadIdx.x == 0) {
        const zero_step_state* st = a.st;
        s_apply = st->apply;
        sk = make_consts(st->beta1, st->beta2, st->beta1_pow, st->beta2_pow, a.lr, a.eps, a.wd, st->clip_coef);
    }
    __syncthreads();
    if (!s_apply) return;  // overflow: the step is skipped
    const AdamConsts k = sk;
    const int nd = ND > 0 ? ND : a.nd;
    for (uint32_t v = blockIdx.x * kThreads + threadIdx.x; v < a.total_v; v += gridDim.x * kThreads) {
        const uint32_t r = v / a.shard_v;
        const uint32_t j = v - r * a.shard_v;
        const size_t o = (size_t)j * kVec;
        const uint64_t out_end = OUT == ZERO_OUT_FULL_REPLICAS ? (uint64_t)(v + 1) * kVec : o + kVec;
        if (!(in_bounds(r + 1, a.bnd.nd) && in_bounds(o + kVec, a.bnd.shard) && in_bounds(out_end, a.bnd.out)))
            continue;
        float g[8], p[8], m[8], w[8];
        ld8(a.gshard[r] + o, g);
        ld8(a.master[r] + o, p);
        ld8(a.m[r] + o, m);
        ld8(a.v[r] + o, w);
        if (all_zero8x3(g, m, w)) {  // e.g. padding, untouched embedding rows
#pragma unroll
            for (int e = 0; e < 8; ++e) adamw1_zero_state(p[e], m[e], w[e], g[e], k);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) adamw1(p[e], m[e], w[e], g[e], k);
        }
        st8(a.master[r] + o, p);
        st8(a.m[r] + o, m);
        st8(a.v[r] + o, w);
        const uint4 h = pack8<F>(p);
        if constexpr (OUT == ZERO_OUT_FULL_REPLICAS) {
            const size_t fo = (size_t)v * kVec;  // ZeRO-1/2: rank-major shard order is flat order
            for (int q = 0; q < nd; ++q) st_stream(a.out[q] + fo, h);
        } else {
            st_stream(a.out[r] + o, h);
        }
    }
}

template <int ND, class F, int OUT>
__global__ void __launch_bounds__(kThreads, 4) fused_kernel(const __grid_constant__ FusedArgs a) {
    __shared__ AdamConsts sk;
    __shared__ float sD;
    const int nd = ND > 0 ? ND : a.nd;
    if (threadIdx.x == 0) {
        const zero_step_state* st = a.st;
        // constants of step t + 1; zero_grad_norm(AFTER_FUSED) advances t afterwards
        sk = make_consts(st->beta1, st->beta2, __dmul_rn(st->beta1_pow, st->beta1),
                         __dmul_rn(st->beta2_pow, st->beta2), a.lr, a.eps, a.wd, 1.0f);
        sD = __fmul_rn((float)nd, st->loss_scale);
    }
    __syncthreads();
    const AdamConsts k = sk;
    const float D = sD;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t gw = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    const uint32_t nw = (gridDim.x * kThreads) >> 5;
    bool bad = false;
    for (uint32_t base = a.seg.v_begin + gw * 32u; base < a.seg.v_end; base += nw * 32u) {
        const uint32_t v = base + lane;
        const bool active = v < a.seg.v_end;
        float g[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) g[e] = 0.0f;
        const uint32_t kk = v - a.seg.seg_v;
        const uint32_t r = kk / a.seg.shard_v;
        const uint32_t j = a.seg.base_v + (kk - r * a.seg.shard_v);
        const size_t o = (size_t)j * kVec;
        const uint64_t out_end = OUT == ZERO_OUT_FULL_REPLICAS ? (uint64_t)(v + 1) * kVec : o + kVec;
        if (active && in_bounds((uint64_t)(v + 1) * kVec, a.bnd.rep) && in_bounds(r + 1, a.bnd.nd) &&
            in_bounds(o + kVec, a.bnd.shard) && in_bounds(out_end, a.bnd.out)) {
            float s[8];
            reduce8<ND, F>(a.rep, nd, v, a.seg.real_end, s);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                bad |= !isfinite(s[e]);
                g[e] = div_rn(s[e], D);
            }
            float p[8], m[8], w[8];
            ld8(a.master[r] + o, p);
            ld8(a.m[r] + o, m);
            ld8(a.v[r] + o, w);
            if (all_zero8x3(g, m, w)) {  // e.g. padding, untouched embedding rows
#pragma unroll
                for (int e = 0; e < 8; ++e) adamw1_zero_state(p[e], m[e], w[e], g[e], k);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) adamw1(p[e], m[e], w[e], g[e], k);
            }
            st8(a.master[r] + o, p);
            st8(a.m[r] + o, m);
            st8(a.v[r] + o, w);
            const uint4 h = pack8<F>(p);
            if constexpr (OUT == ZERO_OUT_FULL_REPLICAS) {
                const size_t fo = (size_t)v * kVec;
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
        const float part = group32_sumsq(g);
        if (active && (lane & 3u) == 0u && in_bounds((v >> 2) + 1, a.bnd.part)) a.partials[v >> 2] = part;
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0u) atomicOr(&a.st->nonfinite, 1);
}

}  // namespace zk

using namespace zero_detail;

template <class Kernel>
static zero_status_t launch_tma(Kernel kern, size_t smem, int64_t tiles, const zk::AdamArgs& a, cudaStream_t s,
                                int threads) {
    static std::mutex mu;
    static std::unordered_map<const void*, int> configured;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!configured.count(reinterpret_cast<const void*>(kern))) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
                return after_launch("zero_adamw_shard_step (shared memory attribute)");
            configured[reinterpret_cast<const void*>(kern)] = 1;
        }
    }
    const int grid = persistent_grid(kern, tiles, smem, threads);
    kern<<<grid, threads, smem, s>>>(a);
    return after_launch("zero_adamw_shard_step");
}

template <int ND, class F, int OUT, int TE, int STAGES, int OST>
static zero_status_t launch_adamw_tma(const zk::AdamArgs& a, cudaStream_t s) {
    const int64_t S = (int64_t)a.shard_v * zk::kVec;
    const int64_t tiles = ((S + TE - 1) / TE) * a.nd;
    // With few bytes per element (16-bit shard output, or at most 4 replicas)
    // the update is bound by instruction latency, and 16 warps per SM beat 8
    // (7B ZeRO-3 shard update 50.2 -> 43.9 ms, before shard outputs moved to
    // the LDG form); with 8 replicas it is bound by bandwidth and 8 warps are
    // faster (10.99 vs 11.38 ms at 1.5B).
    if (OUT == ZERO_OUT_SHARDS || a.nd <= 4)
        return launch_tma(zk::adamw_tma_kernel<ND, F, OUT, TE, STAGES, OST, 512>,
                          zk::AdamTmaSmem<TE, STAGES, OST>::total, tiles, a, s, 512);
    return launch_tma(zk::adamw_tma_kernel<ND, F, OUT, TE, STAGES, OST, 256>, zk::AdamTmaSmem<TE, STAGES, OST>::total,
                      tiles, a, s, 256);
}

// Tile 2048 elements, 4 load stages, 2 output stages (188 KB of shared
// memory, one CTA per SM): on GB300 this shape reaches 98% of the bandwidth a
// plain streaming kernel gets for the 16-byte-read / 28-byte-write mix of the
// 8-replica update.
template <int ND, class F, int OUT>
static zero_status_t launch_adamw_ldg(const zk::AdamArgs& a, cudaStream_t s) {
    auto kern = zk::adamw_ldg_kernel<ND, F, OUT>;
    const int64_t work = ((int64_t)a.total_v + zk::kThreads - 1) / zk::kThreads;
    kern<<<persistent_grid(kern, work), zk::kThreads, 0, s>>>(a);
    return after_launch("zero_adamw_shard_step");
}

// Which form of the update runs (GB300, ms per AdamW call, LDG / TMA): the
// 16-bit shard output of ZeRO-3 moves 30 B per element, too few for the TMA
// pipeline's per-tile barriers (7B block unit 0.965 / 1.204; 350M at N_d = 2,
// 8, 64: 1.67 / 2.07-2.11); full replicas at N_d = 2 also favour LDG (350M
// 1.815 / 1.884), while at N_d = 4..64 the TMA form is equal or faster (350M
// N_d = 4 2.06 / 1.99, N_d = 8 2.53 / 2.49, N_d = 64 9.58 / 9.51; the 1.5B
// block at N_d = 8 0.224 / 0.225).
template <int ND, class F>
static zero_status_t launch_adamw(const zk::AdamArgs& a, int out_kind, cudaStream_t s) {
    const bool ldg = out_kind == ZERO_OUT_SHARDS || a.nd == 2;
    if (ldg) {
        if (out_kind == ZERO_OUT_SHARDS) return launch_adamw_ldg<ND, F, ZERO_OUT_SHARDS>(a, s);
        return launch_adamw_ldg<ND, F, ZERO_OUT_FULL_REPLICAS>(a, s);
    }
    if (out_kind == ZERO_OUT_FULL_REPLICAS) return launch_adamw_tma<ND, F, ZERO_OUT_FULL_REPLICAS, 2048, 4, 2>(a, s);
    return launch_adamw_tma<ND, F, ZERO_OUT_SHARDS, 2048, 4, 2>(a, s);
}

// Resident CTAs per SM for the fused step.  All four that fit are not always
// best: with many replica streams in flight per thread, fewer CTAs keep the
// DRAM pages busier.  GB300, ms per step with 4 / 3 / 2 CTAs per SM:
//   full replicas: N_d=2 (350M) 1.861 / 1.772 / 2.097; N_d=4 2.333 / 2.229 /
//   2.436; N_d=8 (124M) 1.165 / 1.162 / 1.089, (350M) 3.267 / 3.274 / 3.067;
//   N_d=16 5.056 / 4.934 / 5.556; N_d=64 15.95 / 15.82 / 15.71;
//   shard output (ZeRO-3 units): N_d=2 (7B block) 1.381 / 1.387 / 1.571;
//   N_d=8 (350M) 4.840 / 4.762 / 5.031.
// Launches too short to give every thread ~32 vectors at the reduced grid
// keep all four (5M-element buckets, N_d=8: 1.282 / 1.308 / 1.347).
static int64_t fused_ctas_cap(int nd, int out_kind, int64_t nvec) {
    int k = 4;
    if (nd > 1 && out_kind == ZERO_OUT_FULL_REPLICAS) k = nd == 8 ? 2 : 3;
    if (out_kind == ZERO_OUT_SHARDS && nd == 8) k = 3;
    const int64_t sms = sm_count() > 0 ? sm_count() : 1;
    if (nvec < 32 * (int64_t)k * sms * zk::kThreads) k = 4;
    return (int64_t)k * sms;
}

template <int ND, class F>
static zero_status_t launch_fused(const zk::FusedArgs& a, int64_t nvec, int out_kind, cudaStream_t s) {
    const int64_t need = (nvec + zk::kThreads - 1) / zk::kThreads;
    const int64_t cap = fused_ctas_cap(a.nd, out_kind, nvec);
    const int64_t work = need < cap ? need : cap;
    if (out_kind == ZERO_OUT_FULL_REPLICAS) {
        auto kern = zk::fused_kernel<ND, F, ZERO_OUT_FULL_REPLICAS>;
        kern<<<persistent_grid(kern, work), zk::kThreads, 0, s>>>(a);
    } else {
        auto kern = zk::fused_kernel<ND, F, ZERO_OUT_SHARDS>;
        kern<<<persistent_grid(kern, work), zk::kThreads, 0, s>>>(a);
    }
    return after_launch("zero_fused_step");
}

static zero_status_t check_hp(const zero_adamw_hp* hp, const char* what) {
    if (!hp) return fail(ZERO_ERR_INVALID, std::string(what) + ": NULL hyperparameters");
    // eps must stay positive in binary32 too: the update divides by a den of at
    // least eps, and the short path for all-zero elements relies on den > 0
    if (!(hp->lr >= 0.0) || !(hp->eps > 0.0) || !((float)hp->eps > 0.0f) || !(hp->weight_decay >= 0.0))
        return fail(ZERO_ERR_INVALID, std::string(what) +
                                          ": need lr >= 0, eps > 0 (also as a binary32), weight_decay >= 0");
    return ZERO_OK;
}

static zero_status_t check_out(const zero_layout* L, int32_t out_kind, const char* what) {
    if (out_kind != ZERO_OUT_FULL_REPLICAS && out_kind != ZERO_OUT_SHARDS)
        return fail(ZERO_ERR_INVALID, std::string(what) + ": unknown out_kind");
    if (L->stage == 3 && out_kind != ZERO_OUT_SHARDS)
        return fail(ZERO_ERR_STATE, std::string(what) + ": ZeRO-3 writes 16-bit shards only");
    return ZERO_OK;
}

extern "C" zero_status_t zero_adamw_shard_step(const zero_layout* L, const zero_adamw_hp* hp,
                                               float* const* master, float* const* m,
                                               float* const* v, const float* const* grad_shards,
                                               zero_step_state* st, void* const* param16_out,
                                               int32_t out_kind, zero_stream_t stream) {
    clear_error();
    const char* what = "zero_adamw_shard_step";
    if (!L) return fail(ZERO_ERR_INVALID, "zero_adamw_shard_step: NULL layout");
    if (L->stage == 0) return fail(ZERO_ERR_STATE, "zero_adamw_shard_step: stage 0 has no partitioned step");
    zero_status_t rc;
    if ((rc = check_hp(hp, what)) != ZERO_OK) return rc;
    if ((rc = check_out(L, out_kind, what)) != ZERO_OK) return rc;
    const int nd = L->n_d;
    if ((rc = check_ptr_array((const void* const*)master, nd, "zero_adamw_shard_step master")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)m, nd, "zero_adamw_shard_step m")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)v, nd, "zero_adamw_shard_step v")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)grad_shards, nd, "zero_adamw_shard_step grad_shards")) != ZERO_OK)
        return rc;
    if ((rc = check_ptr_array((const void* const*)param16_out, nd, "zero_adamw_shard_step param16_out")) != ZERO_OK)
        return rc;
    if ((rc = check_dev_ptr(st, "zero_adamw_shard_step state")) != ZERO_OK) return rc;

    zk::AdamArgs a{};
    for (int r = 0; r < nd; ++r) {
        a.master[r] = master[r];
        a.m[r] = m[r];
        a.v[r] = v[r];
        a.gshard[r] = grad_shards[r];
        a.out[r] = static_cast<uint16_t*>(param16_out[r]);
    }
    a.st = st;
    a.lr = hp->lr;
    a.eps = hp->eps;
    a.wd = hp->weight_decay;
    a.shard_v = (uint32_t)(L->shard_len / zk::kVec);
    a.total_v = (uint32_t)((int64_t)nd * (L->shard_len / zk::kVec));
    a.nd = nd;
    a.bnd = make_bounds(L, out_kind == ZERO_OUT_FULL_REPLICAS ? L->psi_pad : L->shard_len);
    if (a.total_v == 0) return ZERO_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ZK_DISPATCH(nd, L->dtype, return launch_adamw<ND, F>(a, out_kind, s));
    return ZERO_OK;
}

extern "C" zero_status_t zero_fused_step(const zero_layout* L, int32_t bucket_or_unit,
                                         const zero_adamw_hp* hp, const void* const* grad_replicas,
                                         float* const* master, float* const* m, float* const* v,
                                         zero_step_state* st, void* const* param16_out,
                                         int32_t out_kind, void* workspace, zero_stream_t stream) {
    clear_error();
    const char* what = "zero_fused_step";
    if (!L) return fail(ZERO_ERR_INVALID, "zero_fused_step: NULL layout");
    if (L->stage == 0) return fail(ZERO_ERR_STATE, "zero_fused_step: stage 0 has no partitioned step");
    zero_status_t rc;
    if ((rc = check_hp(hp, what)) != ZERO_OK) return rc;
    if ((rc = check_out(L, out_kind, what)) != ZERO_OK) return rc;
    if (bucket_or_unit < -1 || bucket_or_unit >= (int32_t)L->buckets.size())
        return fail(ZERO_ERR_INVALID, "zero_fused_step: bucket index out of range");
    if (bucket_or_unit == -1 && L->stage == 3 && L->segs.size() > 1)
        return fail(ZERO_ERR_INVALID, "zero_fused_step: ZeRO-3 runs per unit (bucket_or_unit >= 0)");
    const int nd = L->n_d;
    if ((rc = check_ptr_array(grad_replicas, nd, "zero_fused_step grad_replicas")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)master, nd, "zero_fused_step master")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)m, nd, "zero_fused_step m")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)v, nd, "zero_fused_step v")) != ZERO_OK) return rc;
    if ((rc = check_ptr_array((const void* const*)param16_out, nd, "zero_fused_step param16_out")) != ZERO_OK)
        return rc;
    if ((rc = check_dev_ptr(st, "zero_fused_step state")) != ZERO_OK) return rc;
    if ((rc = check_dev_ptr(workspace, "zero_fused_step workspace")) != ZERO_OK) return rc;

    zk::FusedArgs a{};
    for (int r = 0; r < nd; ++r) {
        a.rep[r] = static_cast<const uint16_t*>(grad_replicas[r]);
        a.master[r] = master[r];
        a.m[r] = m[r];
        a.v[r] = v[r];
        a.out[r] = static_cast<uint16_t*>(param16_out[r]);
    }
    a.partials = static_cast<float*>(workspace);
    a.st = st;
    a.lr = hp->lr;
    a.eps = hp->eps;
    a.wd = hp->weight_decay;
    a.nd = nd;
    int64_t begin, end;
    int32_t seg;
    if (bucket_or_unit < 0) {
        begin = 0;
        end = L->psi_pad;
        seg = 0;
    } else {
        begin = L->buckets[bucket_or_unit].first;
        end = L->buckets[bucket_or_unit].second;
        seg = L->bucket_seg[bucket_or_unit];
    }
    a.seg = seg_args(L->segs[seg], begin, end);
    a.bnd = make_bounds(L, out_kind == ZERO_OUT_FULL_REPLICAS ? L->psi_pad : L->shard_len);
    const int64_t nvec = (end - begin) / zk::kVec;
    if (nvec == 0) return ZERO_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ZK_DISPATCH(nd, L->dtype, return launch_fused<ND, F>(a, nvec, out_kind, s));
    return ZERO_OK;
}
