// Step state, the sharding-aware global gradient norm and the step decision.
//
// "ZeRO-3 核心流程：把参数也切开的那一档", 坑 1: gradient clipping must be
// sharding-aware — each rank sees only its 1/N of the norm, and clipping per
// shard gives every rank a different coefficient and silently diverges.  Here
// every reduce-scatter launch leaves one partial sum of squares per 32 flat
// elements; two deterministic passes combine all of them in binary64 in a
// fixed order (independent of bucket sizes, launch shapes and the GPU's SM
// count), so the single coefficient every rank uses is reproducible.
//
// The loss-scale schedule and the overflow skip are not on the pages (config
// reading: fp16 gradients carry a dynamic loss scale; a step whose reduced
// gradient holds an inf or NaN is skipped and the scale halves).
#include <cmath>

#include "zero_launch.h"

namespace zk {

__global__ void state_init_kernel(zero_step_state* st, double beta1, double beta2, float loss_scale,
                                  int32_t dynamic_scale, int32_t growth_interval) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    st->beta1 = beta1;
    st->beta2 = beta2;
    st->beta1_pow = 1.0;
    st->beta2_pow = 1.0;
    st->grad_norm = 0.0;
    st->loss_scale = loss_scale;
    st->clip_coef = 1.0f;
    st->t = 0;
    st->skipped = 0;
    st->good_steps = 0;
    st->growth_interval = growth_interval;
    st->dynamic_scale = dynamic_scale;
    st->nonfinite = 0;
    st->overflow = 0;
    st->apply = 0;
    st->error = 0;
    st->reserved[0] = st->reserved[1] = st->reserved[2] = 0;
}

// Pass 1: block b sums a fixed contiguous range of the partials (fixed
// thread-strided assignment of 16-byte vectors).  Each thread keeps four
// binary32 chains, one per vector lane, each with an error-free TwoSum carry
// (hi + lo holds a chain's sum to ~2^-48 relative; binary64 arithmetic is
// slow on this part), and merges them in lane order; the block then combines
// the threads' hi + lo in binary64 through a fixed pairwise tree.  The range
// length is a multiple of 4 partials (Psi_pad is a multiple of 128), so every
// vector is whole and 16-byte aligned.
__global__ void __launch_bounds__(256) norm_blocks_kernel(const float* __restrict__ partials, uint32_t count,
                                                          double* __restrict__ block_sums) {
    const uint32_t chunk = ((count + gridDim.x - 1) / gridDim.x + 3u) & ~3u;
    const uint32_t b0 = min(count, blockIdx.x * chunk);
    const uint32_t b1 = min(count, b0 + chunk);
    const float4* p4 = reinterpret_cast<const float4*>(partials);
    float hi[4] = {0.0f, 0.0f, 0.0f, 0.0f}, lo[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (uint32_t i = b0 / 4 + threadIdx.x; i < b1 / 4; i += blockDim.x) {
        const float4 x = __ldcs(p4 + i);
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float s, e;
            two_sum(hi[c], xs[c], s, e);
            hi[c] = s;
            lo[c] = __fadd_rn(lo[c], e);
        }
    }
#pragma unroll
    for (int c = 1; c < 4; ++c) {
        float s, e;
        two_sum(hi[0], hi[c], s, e);
        hi[0] = s;
        lo[0] = __fadd_rn(__fadd_rn(lo[0], lo[c]), e);
    }
    __shared__ double sh[256];
    sh[threadIdx.x] = __dadd_rn((double)hi[0], (double)lo[0]);
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) sh[threadIdx.x] = __dadd_rn(sh[threadIdx.x], sh[threadIdx.x + w]);
        __syncthreads();
    }
    if (threadIdx.x == 0) block_sums[blockIdx.x] = sh[0];
}

// Pass 2: one CTA of kNormBlocks threads combines the block sums (fixed tree)
// and updates the step state.
__global__ void __launch_bounds__(zero_detail::kNormBlocks) norm_final_kernel(
        const double* __restrict__ block_sums, zero_step_state* st, double max_norm, int32_t flags) {
    __shared__ double sh[zero_detail::kNormBlocks];
    sh[threadIdx.x] = block_sums[threadIdx.x];
    __syncthreads();
    for (int w = zero_detail::kNormBlocks / 2; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) sh[threadIdx.x] = __dadd_rn(sh[threadIdx.x], sh[threadIdx.x + w]);
        __syncthreads();
    }
    if (threadIdx.x != 0) return;
    const int bad = st->nonfinite != 0;
    st->nonfinite = 0;
    st->overflow = bad;
    const double norm = bad ? (double)INFINITY : __dsqrt_rn(sh[0]);
    st->grad_norm = norm;
    if (flags == ZERO_NORM_AFTER_FUSED) {
        // the fused update already ran with clip 1 and the constants of t + 1
        st->clip_coef = 1.0f;
        st->apply = 1;
        st->t += 1;
        st->beta1_pow = __dmul_rn(st->beta1_pow, st->beta1);
        st->beta2_pow = __dmul_rn(st->beta2_pow, st->beta2);
        st->good_steps += 1;
        return;
    }
    if (bad) {
        st->apply = 0;
        st->clip_coef = 1.0f;
        st->skipped += 1;
        st->good_steps = 0;
        if (st->dynamic_scale) st->loss_scale = fmaxf(1.0f, __fmul_rn(st->loss_scale, 0.5f));
        return;
    }
    float clip = 1.0f;
    if (max_norm > 0.0) clip = __double2float_rn(fmin(1.0, __ddiv_rn(max_norm, __dadd_rn(norm, 1e-6))));
    st->clip_coef = clip;
    st->apply = 1;
    st->t += 1;
    st->beta1_pow = __dmul_rn(st->beta1_pow, st->beta1);
    st->beta2_pow = __dmul_rn(st->beta2_pow, st->beta2);
    st->good_steps += 1;
    if (st->dynamic_scale && st->good_steps >= st->growth_interval) {
        st->loss_scale = __fmul_rn(st->loss_scale, 2.0f);
        st->good_steps = 0;
    }
}

}  // namespace zk

using namespace zero_detail;

extern "C" zero_status_t zero_state_init(zero_step_state* st, double beta1, double beta2,
                                         float loss_scale, int32_t dynamic_scale,
                                         int32_t growth_interval, zero_stream_t stream) {
    clear_error();
    zero_status_t rc;
    if ((rc = check_dev_ptr(st, "zero_state_init state")) != ZERO_OK) return rc;
    if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0))
        return fail(ZERO_ERR_INVALID, "zero_state_init: betas must be in [0, 1)");
    if (!(loss_scale >= 1.0f) || !std::isfinite(loss_scale))
        return fail(ZERO_ERR_INVALID, "zero_state_init: loss_scale must be finite and >= 1");
    if (growth_interval < 1) return fail(ZERO_ERR_INVALID, "zero_state_init: growth_interval must be >= 1");
    zk::state_init_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        st, beta1, beta2, loss_scale, dynamic_scale ? 1 : 0, growth_interval);
    return after_launch("zero_state_init");
}

extern "C" zero_status_t zero_grad_norm(const zero_layout* L, double max_norm, int32_t flags,
                                        zero_step_state* st, void* workspace, zero_stream_t stream) {
    clear_error();
    if (!L) return fail(ZERO_ERR_INVALID, "zero_grad_norm: NULL layout");
    if (L->stage == 0) return fail(ZERO_ERR_STATE, "zero_grad_norm: stage 0 has no partitioned step");
    if (flags != ZERO_NORM_DECIDE && flags != ZERO_NORM_AFTER_FUSED)
        return fail(ZERO_ERR_INVALID, "zero_grad_norm: unknown flags");
    if (std::isnan(max_norm)) return fail(ZERO_ERR_INVALID, "zero_grad_norm: max_norm is NaN");
    zero_status_t rc;
    if ((rc = check_dev_ptr(st, "zero_grad_norm state")) != ZERO_OK) return rc;
    if ((rc = check_dev_ptr(workspace, "zero_grad_norm workspace")) != ZERO_OK) return rc;
    const int64_t count = partials_count(L);
    const int64_t pbytes = ((count * (int64_t)sizeof(float) + 255) / 256) * 256;
    const float* partials = static_cast<const float*>(workspace);
    double* block_sums = reinterpret_cast<double*>(static_cast<char*>(workspace) + pbytes);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    zk::norm_blocks_kernel<<<kNormBlocks, 256, 0, s>>>(partials, (uint32_t)count, block_sums);
    if ((rc = after_launch("zero_grad_norm (pass 1)")) != ZERO_OK) return rc;
    zk::norm_final_kernel<<<1, kNormBlocks, 0, s>>>(block_sums, st, max_norm, flags);
    return after_launch("zero_grad_norm (pass 2)");
}
