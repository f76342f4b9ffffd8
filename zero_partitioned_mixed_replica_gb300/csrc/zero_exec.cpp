// Step executor: one whole ZeRO step as one library call, in the order the
// pages give, from gradients resident in HBM (zero_step) or from gradient
// replicas in host memory (zero_step_from_host).
//
// ZeRO-1/2: reduce-scatter bucket by bucket, last bucket first (backward
// produces the last layers first: the mlqm.cn post "梯度桶化"; reading notes
// "ZeRO: Memory Optimizations Toward Training Trillion Parameter Models"
// §4.1-§4.2) -> global norm and step decision -> sharded AdamW with the
// all-gather fused into its epilogue ("第 5 课：ZeRO 与 FSDP" §3), or the
// fused per-bucket pass when there is neither clipping nor a loss scaler.
// ZeRO-3: forward gathers unit by unit, backward re-gathers each unit in
// reverse and reduce-scatters it (fused: and updates its shard); no all-gather
// at the end of the step ("第 5 课" Fig. 5-1; reading notes §4.3; "ZeRO-3
// 核心流程" §2).
//
// From host memory, each bucket's range (ZeRO-3: each unit's) of every rank's
// replica is copied on two library-owned copy streams, in the order the step
// consumes them, and each bucket's first reading launch waits only for its
// own copies: later buckets cross the host link while earlier ones are
// reduced.  This is the bucketed overlap of the reading notes §4.1-§4.2 (a
// bucket's reduce-scatter starts as soon as backward has filled it), with the
// host link standing in for backward.
#include <cuda_runtime.h>

#include <functional>
#include <mutex>
#include <string>
#include <vector>

#include "zero_internal.h"

using namespace zero_detail;

namespace {

zero_status_t cuda_fail(const char* what, cudaError_t e) {
    return fail(ZERO_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

zero_status_t check_args(const zero_layout* L, const zero_step_args* a, const char* what) {
    const std::string w(what);
    if (!L) return fail(ZERO_ERR_INVALID, w + ": NULL layout");
    if (!a) return fail(ZERO_ERR_INVALID, w + ": NULL arguments");
    if (L->stage == 0) return fail(ZERO_ERR_STATE, w + ": stage 0 has no partitioned step");
    if (a->fused != 0 && a->fused != 1) return fail(ZERO_ERR_INVALID, w + ": fused must be 0 or 1");
    if (a->fused && a->max_norm > 0.0)
        return fail(ZERO_ERR_INVALID, w + ": the fused step cannot clip (use fused = 0)");
    if (!a->fused && !a->grad_shards) return fail(ZERO_ERR_INVALID, w + ": the split step needs grad_shards");
    if (L->stage == 3) {
        if (!a->param16_shards) return fail(ZERO_ERR_INVALID, w + ": ZeRO-3 needs param16_shards");
        if (!a->transient) return fail(ZERO_ERR_INVALID, w + ": ZeRO-3 needs transient buffers");
    } else {
        if (!a->param16_full) return fail(ZERO_ERR_INVALID, w + ": ZeRO-1/2 needs param16_full");
        if (a->fused && a->param16_shards)
            return fail(ZERO_ERR_INVALID, w + ": the fused step writes the full replicas (param16_shards must be NULL)");
    }
    return ZERO_OK;
}

// The step's calls on `s`.  ready(k) runs before the first call that reads the
// gradient replicas of bucket k (ZeRO-3: unit k).
zero_status_t run_step(const zero_layout* L, const zero_step_args* a, zero_stream_t s,
                       const std::function<zero_status_t(int32_t)>& ready) {
    zero_status_t rc;
    const int32_t nb = (int32_t)L->buckets.size();
    if (L->stage == 3) {
        const int32_t U = (int32_t)L->segs.size();
        for (int32_t u = 0; u < U; ++u)  // forward
            if ((rc = zero_stage3_gather_layer(L, u, (const void* const*)a->param16_shards, a->transient, s)) != ZERO_OK)
                return rc;
        for (int32_t u = U - 1; u >= 0; --u) {  // backward
            if ((rc = zero_stage3_gather_layer(L, u, (const void* const*)a->param16_shards, a->transient, s)) != ZERO_OK)
                return rc;
            if ((rc = ready(u)) != ZERO_OK) return rc;
            rc = a->fused ? zero_fused_step(L, u, a->hp, a->grad_replicas, a->master, a->m, a->v, a->state,
                                            a->param16_shards, ZERO_OUT_SHARDS, a->workspace, s)
                          : zero_reduce_scatter(L, u, a->grad_replicas, a->grad_shards, a->state, a->workspace, s);
            if (rc != ZERO_OK) return rc;
        }
        if (a->fused) return zero_grad_norm(L, 0.0, ZERO_NORM_AFTER_FUSED, a->state, a->workspace, s);
        if ((rc = zero_grad_norm(L, a->max_norm, ZERO_NORM_DECIDE, a->state, a->workspace, s)) != ZERO_OK) return rc;
        return zero_adamw_shard_step(L, a->hp, a->master, a->m, a->v, (const float* const*)a->grad_shards, a->state,
                                     a->param16_shards, ZERO_OUT_SHARDS, s);
    }
    if (a->fused) {
        if (a->per_bucket) {
            for (int32_t b = nb - 1; b >= 0; --b) {
                if ((rc = ready(b)) != ZERO_OK) return rc;
                if ((rc = zero_fused_step(L, b, a->hp, a->grad_replicas, a->master, a->m, a->v, a->state,
                                          a->param16_full, ZERO_OUT_FULL_REPLICAS, a->workspace, s)) != ZERO_OK)
                    return rc;
            }
        } else {
            for (int32_t b = nb - 1; b >= 0; --b)
                if ((rc = ready(b)) != ZERO_OK) return rc;
            if ((rc = zero_fused_step(L, -1, a->hp, a->grad_replicas, a->master, a->m, a->v, a->state,
                                      a->param16_full, ZERO_OUT_FULL_REPLICAS, a->workspace, s)) != ZERO_OK)
                return rc;
        }
        return zero_grad_norm(L, 0.0, ZERO_NORM_AFTER_FUSED, a->state, a->workspace, s);
    }
    for (int32_t b = nb - 1; b >= 0; --b) {
        if ((rc = ready(b)) != ZERO_OK) return rc;
        if ((rc = zero_reduce_scatter(L, b, a->grad_replicas, a->grad_shards, a->state, a->workspace, s)) != ZERO_OK)
            return rc;
    }
    if ((rc = zero_grad_norm(L, a->max_norm, ZERO_NORM_DECIDE, a->state, a->workspace, s)) != ZERO_OK) return rc;
    if (!a->param16_shards)
        return zero_adamw_shard_step(L, a->hp, a->master, a->m, a->v, (const float* const*)a->grad_shards, a->state,
                                     a->param16_full, ZERO_OUT_FULL_REPLICAS, s);
    if ((rc = zero_adamw_shard_step(L, a->hp, a->master, a->m, a->v, (const float* const*)a->grad_shards, a->state,
                                    a->param16_shards, ZERO_OUT_SHARDS, s)) != ZERO_OK)
        return rc;
    return zero_allgather_params(L, (const void* const*)a->param16_shards, a->param16_full, s);
}

// Library-owned copy streams and events of one device, created at the first
// host-input step on it and kept until the process exits.
struct CopyStreams {
    cudaStream_t cs[2] = {nullptr, nullptr};
    cudaEvent_t start = nullptr;
    std::vector<cudaEvent_t> ev;  // two per bucket: one per copy stream
};

std::mutex g_copy_mu;
CopyStreams g_copy[64];

zero_status_t copy_streams(int dev, size_t n_events, CopyStreams** out) {
    CopyStreams& c = g_copy[dev];
    cudaError_t e;
    for (int i = 0; i < 2; ++i)
        if (!c.cs[i] && (e = cudaStreamCreateWithFlags(&c.cs[i], cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail("zero_step_from_host: copy stream", e);
    if (!c.start && (e = cudaEventCreateWithFlags(&c.start, cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail("zero_step_from_host: event", e);
    while (c.ev.size() < n_events) {
        cudaEvent_t x = nullptr;
        if ((e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail("zero_step_from_host: event", e);
        c.ev.push_back(x);
    }
    *out = &c;
    return ZERO_OK;
}

}  // namespace

extern "C" zero_status_t zero_step(const zero_layout* L, const zero_step_args* a, zero_stream_t stream) {
    clear_error();
    zero_status_t rc = check_args(L, a, "zero_step");
    if (rc != ZERO_OK) return rc;
    return run_step(L, a, stream, [](int32_t) { return ZERO_OK; });
}

extern "C" zero_status_t zero_step_from_host(const zero_layout* L, const zero_step_args* a,
                                             const void* const* host_grads, int64_t chunk_elems,
                                             void* host_state, zero_stream_t stream) {
    clear_error();
    zero_status_t rc = check_args(L, a, "zero_step_from_host");
    if (rc != ZERO_OK) return rc;
    if (!host_grads) return fail(ZERO_ERR_INVALID, "zero_step_from_host: NULL host gradient array");
    if (!a->grad_replicas) return fail(ZERO_ERR_INVALID, "zero_step_from_host: NULL device gradient array");
    for (int r = 0; r < L->n_d; ++r) {
        if (!host_grads[r]) return fail(ZERO_ERR_INVALID, "zero_step_from_host: NULL host gradient replica");
        if (!a->grad_replicas[r]) return fail(ZERO_ERR_INVALID, "zero_step_from_host: NULL device gradient replica");
    }
    if (chunk_elems <= 0) chunk_elems = (int64_t)1 << 27;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("zero_step_from_host", e);
    if (dev < 0 || dev >= 64) return fail(ZERO_ERR_CUDA, "zero_step_from_host: device index >= 64");
    const int32_t nb = (int32_t)L->buckets.size();
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(g_copy_mu);  // the events are reused by every call on this device
    CopyStreams* c = nullptr;
    if ((rc = copy_streams(dev, 2 * (size_t)nb, &c)) != ZERO_OK) return rc;
    // the previous step on `stream` has finished reading the replicas before they are overwritten
    if ((e = cudaEventRecord(c->start, s)) != cudaSuccess) return cuda_fail("zero_step_from_host: record", e);
    for (int i = 0; i < 2; ++i)
        if ((e = cudaStreamWaitEvent(c->cs[i], c->start, 0)) != cudaSuccess)
            return cuda_fail("zero_step_from_host: wait", e);
    // copies in the order the step consumes the buckets (units): last first
    const size_t esz = sizeof(uint16_t);
    int64_t i = 0;
    for (int32_t k = nb - 1; k >= 0; --k) {
        const int64_t lo = L->buckets[k].first, hi = L->buckets[k].second;
        for (int r = 0; r < L->n_d; ++r) {
            for (int64_t off = lo; off < hi; off += chunk_elems, ++i) {
                const int64_t n = (hi - off) < chunk_elems ? (hi - off) : chunk_elems;
                e = cudaMemcpyAsync(static_cast<char*>(const_cast<void*>(a->grad_replicas[r])) + off * esz,
                                    static_cast<const char*>(host_grads[r]) + off * esz, (size_t)n * esz,
                                    cudaMemcpyHostToDevice, c->cs[i % 2]);
                if (e != cudaSuccess) return cuda_fail("zero_step_from_host: host-to-device copy", e);
            }
        }
        for (int q = 0; q < 2; ++q)
            if ((e = cudaEventRecord(c->ev[2 * k + q], c->cs[q])) != cudaSuccess)
                return cuda_fail("zero_step_from_host: record", e);
    }
    rc = run_step(L, a, stream, [&](int32_t k) -> zero_status_t {
        for (int q = 0; q < 2; ++q) {
            cudaError_t w = cudaStreamWaitEvent(s, c->ev[2 * k + q], 0);
            if (w != cudaSuccess) return cuda_fail("zero_step_from_host: wait", w);
        }
        return ZERO_OK;
    });
    if (rc != ZERO_OK) return rc;
    if (host_state) {
        e = cudaMemcpyAsync(host_state, a->state, sizeof(zero_step_state), cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail("zero_step_from_host: state read-back", e);
    }
    return ZERO_OK;
}
