// Device-side building blocks of libzero (sm_103a).
//
// All floating-point arithmetic of the step goes through explicitly rounded
// intrinsics (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn, ...), so no
// multiply-add is ever contracted and every operation is one IEEE-754
// binary32 operation, round to nearest even.  The library is additionally
// compiled with -fmad=false.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "zero.h"

namespace zk {

constexpr int kThreads = 256;      // threads per CTA of the streaming kernels
constexpr int kVec = 8;            // 16-bit elements per 16-byte vector
constexpr int kMaxRanks = ZERO_MAX_RANKS;

// Extents (elements) of the buffers a launch touches, from the layout; the
// bounds-checked build tests every global access against them.
struct Bounds {
    uint64_t rep;    // each 16-bit gradient replica or fp32 accumulator: Psi_pad
    uint64_t shard;  // each fp32 shard (master, m, v, reduced gradient): S
    uint64_t out;    // each 16-bit output: Psi_pad, S, or a transient's unit size
    uint64_t part;   // norm partials: Psi_pad / 32
    uint64_t src;    // each 16-bit shard a gather reads: S
    uint32_t nd;     // rank index bound
    uint32_t pad0;
};

#ifdef ZK_CHECKED
constexpr bool kChecked = true;
// Accesses skipped by the checks, one counter per translation unit (the host
// sums them, zero_bounds_violations).
static __device__ unsigned long long zk_bounds_hits;
#else
constexpr bool kChecked = false;
#endif

// True if [.., end) lies inside an extent of `lim` elements.  The checked
// build counts and reports a miss (the caller skips the access); the normal
// build compiles to `true`.
__device__ __forceinline__ bool in_bounds(uint64_t end, uint64_t lim) {
#ifdef ZK_CHECKED
    if (end > lim) {
        atomicAdd(&zk_bounds_hits, 1ull);
        return false;
    }
#else
    (void)end;
    (void)lim;
#endif
    return true;
}

// ----------------------------------------------------------------------------
// 16-bit formats
// ----------------------------------------------------------------------------
struct Bf16 {
    static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
    static __device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
    }
    static __device__ __forceinline__ uint16_t enc1(float a) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(a));
    }
    static __device__ __forceinline__ float dec1(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
};

struct Fp16 {
    static __device__ __forceinline__ float lo(uint32_t w) {
        return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
    }
    static __device__ __forceinline__ float hi(uint32_t w) {
        return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
    }
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        return (uint32_t)__half_as_ushort(__float2half_rn(a)) |
               ((uint32_t)__half_as_ushort(__float2half_rn(b)) << 16);
    }
    static __device__ __forceinline__ uint16_t enc1(float a) { return __half_as_ushort(__float2half_rn(a)); }
    static __device__ __forceinline__ float dec1(uint16_t h) { return __half2float(__ushort_as_half(h)); }
};

template <class F>
__device__ __forceinline__ void unpack8(const uint4& x, float (&o)[8]) {
    o[0] = F::lo(x.x); o[1] = F::hi(x.x);
    o[2] = F::lo(x.y); o[3] = F::hi(x.y);
    o[4] = F::lo(x.z); o[5] = F::hi(x.z);
    o[6] = F::lo(x.w); o[7] = F::hi(x.w);
}

template <class F>
__device__ __forceinline__ uint4 pack8(const float (&p)[8]) {
    uint4 r;
    r.x = F::pack(p[0], p[1]);
    r.y = F::pack(p[2], p[3]);
    r.z = F::pack(p[4], p[5]);
    r.w = F::pack(p[6], p[7]);
    return r;
}

// ----------------------------------------------------------------------------
// Memory access: every big buffer is streamed once per step.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ float4 ld_stream(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_stream(uint16_t* p, uint4 v) { __stcs(reinterpret_cast<uint4*>(p), v); }
__device__ __forceinline__ void st_stream(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

// 8 consecutive floats as one 32-byte access (sm_100+ 256-bit vector form),
// cache-streaming; p must be 32-byte aligned.
__device__ __forceinline__ void ld8(const float* p, float (&o)[8]) {
    asm volatile("ld.global.cs.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(o[0]), "=f"(o[1]), "=f"(o[2]), "=f"(o[3]), "=f"(o[4]), "=f"(o[5]), "=f"(o[6]), "=f"(o[7])
                 : "l"(p));
}
__device__ __forceinline__ void st8(float* p, const float (&o)[8]) {
    asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(o[0]), "f"(o[1]), "f"(o[2]),
                 "f"(o[3]), "f"(o[4]), "f"(o[5]), "f"(o[6]), "f"(o[7])
                 : "memory");
}

// 16 consecutive 16-bit values as one 32-byte access; p 32-byte aligned.
__device__ __forceinline__ void ld16h(const uint16_t* p, uint32_t (&w)[8]) {
    asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}

template <class F>
__device__ __forceinline__ void unpack16(const uint32_t (&w)[8], float (&o)[16]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        o[2 * k] = F::lo(w[k]);
        o[2 * k + 1] = F::hi(w[k]);
    }
}

// 16-element form of reduce8 (compile-time ND only): all N_d loads are issued
// before the rank-order sum.
template <int ND, class F>
__device__ __forceinline__ void reduce16(const uint16_t* const* rep, uint32_t v16, int64_t real_end,
                                         float (&s)[16]) {
    const int64_t i0 = (int64_t)v16 * 16;
    if (i0 + 16 <= real_end) {
        uint32_t w[ND][8];
#pragma unroll
        for (int r = 0; r < ND; ++r) ld16h(rep[r] + i0, w[r]);
        unpack16<F>(w[0], s);
#pragma unroll
        for (int r = 1; r < ND; ++r) {
            float t[16];
            unpack16<F>(w[r], t);
#pragma unroll
            for (int e = 0; e < 16; ++e) s[e] = __fadd_rn(s[e], t[e]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) s[e] = 0.0f;
        for (int e = 0; e < 16; ++e) {
            if (i0 + e >= real_end) break;
            float acc = F::dec1(rep[0][i0 + e]);
            for (int r = 1; r < ND; ++r) acc = __fadd_rn(acc, F::dec1(rep[r][i0 + e]));
            s[e] = acc;
        }
    }
}

// ----------------------------------------------------------------------------
// Gradient reduction: s = x_0 + x_1 + ... in rank order; padding reads 0.
// ND > 0: compile-time rank count; ND == 0: runtime `nd`.
// ----------------------------------------------------------------------------
template <int ND, class F>
__device__ __forceinline__ void reduce8(const uint16_t* const* rep, int nd, uint32_t v,
                                        int64_t real_end, float (&s)[8]) {
    const int64_t i0 = (int64_t)v * kVec;
    const int n = ND > 0 ? ND : nd;
    if (i0 + kVec <= real_end) {
        if constexpr (ND > 0) {
            uint4 x[ND];
#pragma unroll
            for (int r = 0; r < ND; ++r) x[r] = ld_stream(rep[r] + i0);
            unpack8<F>(x[0], s);
#pragma unroll
            for (int r = 1; r < ND; ++r) {
                float t[8];
                unpack8<F>(x[r], t);
#pragma unroll
                for (int e = 0; e < 8; ++e) s[e] = __fadd_rn(s[e], t[e]);
            }
        } else {
            uint4 x0 = ld_stream(rep[0] + i0);
            unpack8<F>(x0, s);
            int r = 1;
            for (; r + 4 <= n; r += 4) {
                uint4 x[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) x[k] = ld_stream(rep[r + k] + i0);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float t[8];
                    unpack8<F>(x[k], t);
#pragma unroll
                    for (int e = 0; e < 8; ++e) s[e] = __fadd_rn(s[e], t[e]);
                }
            }
            for (; r < n; ++r) {
                float t[8];
                unpack8<F>(ld_stream(rep[r] + i0), t);
#pragma unroll
                for (int e = 0; e < 8; ++e) s[e] = __fadd_rn(s[e], t[e]);
            }
        }
    } else {
        // Vector that reaches into (or lies in) the segment's padding: element
        // loads, padding contributes exactly 0.
#pragma unroll
        for (int e = 0; e < 8; ++e) s[e] = 0.0f;
        for (int e = 0; e < 8; ++e) {
            if (i0 + e >= real_end) break;
            float acc = F::dec1(rep[0][i0 + e]);
            for (int r = 1; r < n; ++r) acc = __fadd_rn(acc, F::dec1(rep[r][i0 + e]));
            s[e] = acc;
        }
    }
}

// ----------------------------------------------------------------------------
// Sum of squares with an error-free transformation (Knuth's TwoSum and the
// FMA-based TwoProduct; Ogita, Rump and Oishi, "Accurate Sum and Dot
// Product", SIAM J. Sci. Comput. 26(6), 2005): (hi, lo) carries the running
// sum and its accumulated rounding errors.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void acc_sq(float x, float& hi, float& lo) {
    float p = __fmul_rn(x, x);
    float pe = __fmaf_rn(x, x, -p);  // exact remainder x*x - p
    float s, e;
    two_sum(hi, p, s, e);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(e, pe));
}

// Combine with the partner lane `mask` away; symmetric, so both lanes end
// with the same bits.
__device__ __forceinline__ void combine_lanes(float& hi, float& lo, int mask) {
    float ohi = __shfl_xor_sync(0xFFFFFFFFu, hi, mask);
    float olo = __shfl_xor_sync(0xFFFFFFFFu, lo, mask);
    float s, e;
    two_sum(hi, ohi, s, e);
    hi = s;
    lo = __fadd_rn(__fadd_rn(lo, olo), e);
}

// 32-element group partial of 4 consecutive lanes (8 elements each).  All 32
// lanes must call it.  Returns the group's sum of squares rounded once.
__device__ __forceinline__ float group32_sumsq(const float (&g)[8]) {
    float hi = 0.0f, lo = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc_sq(g[e], hi, lo);
    combine_lanes(hi, lo, 1);
    combine_lanes(hi, lo, 2);
    return __fadd_rn(hi, lo);
}

// ----------------------------------------------------------------------------
// AdamW, decoupled weight decay, one rounding per operation.
// ----------------------------------------------------------------------------
struct AdamConsts {
    float decay, b1, b2, omb1, omb2, eps, step_size, sqrt_bc2, clip;
};

// Constants of the step whose bias corrections are beta1^t = b1p and
// beta2^t = b2p, computed in binary64 (IEEE division and square root) and
// rounded once to binary32.
__device__ __forceinline__ AdamConsts make_consts(double beta1, double beta2, double b1p, double b2p,
                                                  double lr, double eps, double wd, float clip) {
    AdamConsts k;
    k.decay = __double2float_rn(__dsub_rn(1.0, __dmul_rn(lr, wd)));
    k.b1 = __double2float_rn(beta1);
    k.b2 = __double2float_rn(beta2);
    k.omb1 = __double2float_rn(__dsub_rn(1.0, beta1));
    k.omb2 = __double2float_rn(__dsub_rn(1.0, beta2));
    k.eps = __double2float_rn(eps);
    k.step_size = __double2float_rn(__ddiv_rn(lr, __dsub_rn(1.0, b1p)));
    k.sqrt_bc2 = __double2float_rn(__dsqrt_rn(__dsub_rn(1.0, b2p)));
    k.clip = clip;
    return k;
}

// x / y, IEEE round-to-nearest-even, with a zero x over a positive y (+inf
// included) answered directly: a zero with x's sign.  The rounded division
// runs on a stand-in numerator of 1 in those lanes, so it never takes its
// zero-operand path, which is slow on GB300; any other x, or y <= 0 or NaN,
// goes through the rounded division.  Used for the division by N_d *
// loss_scale, where a gradient summed to zero (padding, untouched embedding
// rows) is common.
__device__ __forceinline__ float div_rn(float x, float y) {
    const bool z = (x == 0.0f) && (y > 0.0f);
    const float q = __fdiv_rn(z ? 1.0f : x, y);
    return z ? x : q;
}

// True when every value is +0 or -0 (bit patterns OR-ed, sign bits masked).
__device__ __forceinline__ bool all_zero8x3(const float (&a)[8], const float (&b)[8], const float (&c)[8]) {
    uint32_t x = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) x |= __float_as_uint(a[e]) | __float_as_uint(b[e]) | __float_as_uint(c[e]);
    return (x & 0x7FFFFFFFu) == 0u;
}

// One element's AdamW update (binary32, one rounding per operation, no FMA).
__device__ __forceinline__ void adamw1(float& p, float& m, float& v, float g, const AdamConsts& k) {
    const float gc = __fmul_rn(g, k.clip);
    const float p1 = __fmul_rn(p, k.decay);
    const float mn = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.omb1, gc));
    const float vn = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.omb2, __fmul_rn(gc, gc)));
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(vn), k.sqrt_bc2), k.eps);
    p = __fsub_rn(p1, __fmul_rn(k.step_size, __fdiv_rn(mn, den)));
    m = mn;
    v = vn;
}

// The same update for an element whose g, m and v are all zero (of either
// sign): the new m and v are zeros, den = eps > 0 and m / den is m itself (a
// zero over a positive number), so p = p1 - step_size * m exactly, without
// the rounded square root and division.  Their zero-operand paths are slow on
// GB300: a 7B ZeRO-3 step with all-zero gradients took 55.1 against 42.2 ms.
__device__ __forceinline__ void adamw1_zero_state(float& p, float& m, float& v, float g, const AdamConsts& k) {
    const float gc = __fmul_rn(g, k.clip);
    const float p1 = __fmul_rn(p, k.decay);
    const float mn = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.omb1, gc));
    const float vn = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.omb2, __fmul_rn(gc, gc)));
    p = __fsub_rn(p1, __fmul_rn(k.step_size, mn));
    m = mn;
    v = vn;
}

// ----------------------------------------------------------------------------
// Bulk asynchronous copies (TMA, 1-D form) and mbarriers, inline PTX.
// Every wait on an mbarrier is bounded in time: once kWaitLimitNs of the
// global timer have passed (or, as a backstop, kWaitMaxPolls polls) the wait
// gives up, and the caller records ZERO_DEVERR_WAIT_TIMEOUT in the step state
// and unwinds.  A poll (mbarrier.try_wait) may itself suspend the thread for
// a system-dependent time, so a poll count alone does not bound the time.
// ----------------------------------------------------------------------------
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
constexpr uint32_t kWaitMaxPolls = 1u << 26;
constexpr int32_t ZERO_DEVERR_WAIT_TIMEOUT = 1;
// While unwinding after ZERO_DEVERR_WAIT_TIMEOUT, a CTA waits up to
// kDrainTries bounded waits for each of its loads still in flight; one that
// never lands is reported with this bit.
constexpr int32_t ZERO_DEVERR_DRAIN_TIMEOUT = 2;
constexpr int kDrainTries = 4;

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (bulk stores issued after the next barrier read them).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait; false if the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;  // the common case: no timer read
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; i < kWaitMaxPolls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
    return false;
}
// global -> this CTA's shared memory, completion counted on `bar` (bytes).
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// shared -> global, tracked by bulk async-groups.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src_smem)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ----------------------------------------------------------------------------
// Kernel arguments (passed by value as __grid_constant__ parameters).
// Vector indices count 8-element vectors of the flat buffer (32-bit: the
// layout rejects Psi_pad >= 2^34).
// ----------------------------------------------------------------------------
struct SegArgs {
    uint32_t v_begin, v_end;  // flat vector range processed by this launch
    uint32_t seg_v;           // segment offset (vectors)
    uint32_t shard_v;         // S_u / 8
    uint32_t base_v;          // shard_base / 8
    uint32_t pad0;
    int64_t real_end;         // flat index where the segment's padding starts
};

struct RsArgs {
    const uint16_t* rep[kMaxRanks];
    float* gshard[kMaxRanks];
    float* partials;
    zero_step_state* st;
    SegArgs seg;
    Bounds bnd;
    int32_t nd;
    int32_t n_micro;  // micro-batches of the step (1: plain reduce-scatter)
};

// Reduce-scatter modes: plain, and the first / middle / last micro-batch of
// an accumulated step.
enum { RS_PLAIN = 0, RS_FIRST = 1, RS_MIDDLE = 2, RS_LAST = 3 };

struct AccumArgs {
    const uint16_t* rep[kMaxRanks];
    float* acc[kMaxRanks];
    Bounds bnd;
    uint32_t v_per_rank;  // Psi_pad / 8
    int64_t real_end;     // padding starts here
    int32_t nd;
};

struct RsAccArgs {
    const float* acc[kMaxRanks];
    float* gshard[kMaxRanks];
    float* partials;
    zero_step_state* st;
    SegArgs seg;
    Bounds bnd;
    int32_t nd;
    int32_t n_micro;
};

struct AdamArgs {
    float* master[kMaxRanks];
    float* m[kMaxRanks];
    float* v[kMaxRanks];
    const float* gshard[kMaxRanks];
    uint16_t* out[kMaxRanks];
    zero_step_state* st;
    Bounds bnd;
    double lr, eps, wd;
    uint32_t shard_v;   // per-rank shard length / 8
    uint32_t total_v;   // nd * shard_v
    int32_t nd;
};

struct FusedArgs {
    const uint16_t* rep[kMaxRanks];
    float* master[kMaxRanks];
    float* m[kMaxRanks];
    float* v[kMaxRanks];
    uint16_t* out[kMaxRanks];
    float* partials;
    zero_step_state* st;
    Bounds bnd;
    double lr, eps, wd;
    SegArgs seg;
    int32_t nd;
};

struct GatherArgs {
    const uint16_t* src[kMaxRanks];
    uint16_t* dst[kMaxRanks];
    Bounds bnd;
    uint32_t shard_v;   // S_u / 8
    uint32_t base_v;    // shard_base / 8
    int64_t n_elems;    // elements per destination (real_u, or Psi_pad)
    int32_t nd;
};

}  // namespace zk
