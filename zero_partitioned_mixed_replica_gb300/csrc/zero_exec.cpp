// Step executor: one whole ZeRO step as one library call, in the order the
// pages give, from gradients resident in HBM (zero_step), from gradient
// replicas in host memory (zero_step_from_host), or one micro-batch of an
// accumulated step (zero_micro_step); plus the launch tracing of the calls it
// issues.
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
// host link standing in for backward.  With overlap_previous, consecutive
// host-input steps also overlap: a step's copies wait only for the previous
// step's last replica-reading launch, not for its norm and update.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
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

zero_status_t check_ptrs(const void* const* arr, int n, const std::string& what) {
    if (!arr) return ZERO_OK;  // presence is checked per stage
    for (int i = 0; i < n; ++i) {
        if (!arr[i]) return fail(ZERO_ERR_INVALID, what + ": NULL device pointer");
        if (reinterpret_cast<uintptr_t>(arr[i]) & 255u)
            return fail(ZERO_ERR_ALIGN, what + ": device pointer not 256-byte aligned");
    }
    return ZERO_OK;
}

zero_status_t check_args(const zero_layout* L, const zero_step_args* a, const char* what) {
    const std::string w(what);
    if (!L) return fail(ZERO_ERR_INVALID, w + ": NULL layout");
    if (!a) return fail(ZERO_ERR_INVALID, w + ": NULL arguments");
    if (L->stage == 0) return fail(ZERO_ERR_STATE, w + ": stage 0 has no partitioned step");
    if (a->fused != 0 && a->fused != 1) return fail(ZERO_ERR_INVALID, w + ": fused must be 0 or 1");
    if (a->overlap_previous != 0 && a->overlap_previous != 1)
        return fail(ZERO_ERR_INVALID, w + ": overlap_previous must be 0 or 1");
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
    if (!a->hp) return fail(ZERO_ERR_INVALID, w + ": NULL hyperparameters");
    if (!a->grad_replicas || !a->master || !a->m || !a->v)
        return fail(ZERO_ERR_INVALID, w + ": NULL pointer array");
    const int n = L->n_d;
    zero_status_t rc;
    if ((rc = check_ptrs(a->grad_replicas, n, w + " grad_replicas")) != ZERO_OK) return rc;
    if ((rc = check_ptrs((const void* const*)a->master, n, w + " master")) != ZERO_OK) return rc;
    if ((rc = check_ptrs((const void* const*)a->m, n, w + " m")) != ZERO_OK) return rc;
    if ((rc = check_ptrs((const void* const*)a->v, n, w + " v")) != ZERO_OK) return rc;
    if ((rc = check_ptrs((const void* const*)a->grad_shards, n, w + " grad_shards")) != ZERO_OK) return rc;
    if ((rc = check_ptrs((const void* const*)a->param16_full, n, w + " param16_full")) != ZERO_OK) return rc;
    if ((rc = check_ptrs((const void* const*)a->param16_shards, n, w + " param16_shards")) != ZERO_OK) return rc;
    if ((rc = check_ptrs((const void* const*)a->transient, n, w + " transient")) != ZERO_OK) return rc;
    if (a->transient2 && L->stage != 3) return fail(ZERO_ERR_INVALID, w + ": transient2 is for ZeRO-3 only");
    if (a->unit_hook && L->stage != 3) return fail(ZERO_ERR_INVALID, w + ": unit_hook is for ZeRO-3 only");
    if ((rc = check_ptrs((const void* const*)a->transient2, n, w + " transient2")) != ZERO_OK) return rc;
    const void* one[2] = {a->state, a->workspace};
    if (!a->state || !a->workspace) return fail(ZERO_ERR_INVALID, w + ": NULL state or workspace");
    return check_ptrs(one, 2, w + " state/workspace");
}

// ---------------------------------------------------------------------------
// Launch tracing: with tracing on, every call the executor issues is
// bracketed by two timing events recorded on the stream it is issued on
// (not while that stream is being captured into a graph).
// ---------------------------------------------------------------------------
// At most this many calls are kept between reads; later calls run untraced.
constexpr size_t kTraceMaxRecords = (size_t)1 << 20;

struct TraceRecord {
    int32_t kind;
    int32_t dev;
    cudaStream_t stream;
    cudaEvent_t e0, e1;
};
std::mutex g_trace_mu;
std::atomic<int32_t> g_trace_on{0};
std::vector<TraceRecord> g_trace;
std::vector<cudaEvent_t> g_trace_free[64];

bool trace_take(int dev, cudaEvent_t* e) {
    auto& pool = g_trace_free[dev];
    if (!pool.empty()) {
        *e = pool.back();
        pool.pop_back();
        return true;
    }
    return cudaEventCreate(e) == cudaSuccess;
}

template <class Call>
zero_status_t traced(int32_t kind, cudaStream_t st, Call&& call) {
    if (!g_trace_on.load(std::memory_order_relaxed)) return call();
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    int dev = 0;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone ||
        cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return call();
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_trace_mu);
        if (g_trace.size() >= kTraceMaxRecords || !trace_take(dev, &e0)) return call();
        if (!trace_take(dev, &e1)) {
            g_trace_free[dev].push_back(e0);
            return call();
        }
    }
    cudaEventRecord(e0, st);
    const zero_status_t rc = call();
    cudaEventRecord(e1, st);
    std::lock_guard<std::mutex> lock(g_trace_mu);
    g_trace.push_back({kind, dev, st, e0, e1});
    return rc;
}

// ---------------------------------------------------------------------------
// Per-device resources of the executor, created at first use and kept until
// the process exits: the extra streams that bucket launches rotate over, with their
// fork/join events, and the host-input copy streams with their events.  One
// lock per device serialises the calls that use them.
// ---------------------------------------------------------------------------
// Streams that short bucket launches rotate over (the caller's plus
// kLanes - 1 of the library's).  GB300, ms per step eager / from a CUDA
// graph.  GPT-2 small ZeRO-1, 25 buckets of 5M elements: 2 lanes 1.081 /
// 1.074, 3 lanes 1.065 / 1.052, 4 lanes 1.054 / 1.051; 4, 6 and 8 lanes
// equal on another box.  350M layout, N_d = 8, 3549 buckets of 1e5 elements:
// 4 lanes 11.39 / 9.84, 6 lanes 8.39 / 7.06, 8 lanes 8.37 / 5.79.
#ifndef ZK_BUCKET_LANES
#define ZK_BUCKET_LANES 8
#endif
constexpr int kLanes = ZK_BUCKET_LANES;
static_assert(kLanes >= 2, "the executor needs a second stream");

struct DeviceRes {
    std::mutex mu;
    cudaStream_t aux[kLanes - 1] = {};
    cudaEvent_t fork = nullptr, join[kLanes - 1] = {};
    cudaStream_t cs[2] = {nullptr, nullptr};
    cudaEvent_t start = nullptr;
    std::vector<cudaEvent_t> ev;  // two per bucket: one per copy stream
    // Recorded by zero_step_from_host after its last launch that reads the
    // device replicas; released_ok says that call succeeded outside a capture
    // and no other executor call has run on the device since.  The call's
    // stream and device replica pointers: a later call takes the early gate
    // only with the same ones (another set of replicas was last read by a
    // step this event does not follow).
    cudaEvent_t released = nullptr;
    bool released_ok = false;
    cudaStream_t released_stream = nullptr;
    std::vector<const void*> released_grads;
};
DeviceRes g_res[64];

zero_status_t current_res(DeviceRes** out, const char* what) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(what, e);
    if (dev < 0 || dev >= 64) return fail(ZERO_ERR_CUDA, std::string(what) + ": device index >= 64");
    *out = &g_res[dev];
    return ZERO_OK;
}

zero_status_t make_stream(cudaStream_t* s, const char* what) {
    if (*s) return ZERO_OK;
    cudaError_t e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(what, e);
}

zero_status_t make_event(cudaEvent_t* ev, const char* what) {
    if (*ev) return ZERO_OK;
    cudaError_t e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(what, e);
}

zero_status_t step_res(DeviceRes& R, const char* what) {
    zero_status_t rc;
    for (int i = 0; i < kLanes - 1; ++i) {
        if ((rc = make_stream(&R.aux[i], what)) != ZERO_OK) return rc;
        if ((rc = make_event(&R.join[i], what)) != ZERO_OK) return rc;
    }
    return make_event(&R.fork, what);
}

zero_status_t wait_on(cudaStream_t waiter, cudaEvent_t ev, cudaStream_t recorder, const char* what) {
    cudaError_t e = cudaEventRecord(ev, recorder);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(waiter, ev, 0);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(what, e);
}

// The device's extra streams, forked from `s` (they wait for the work queued
// on `s`) and joined back (`s` waits for them) explicitly or, if a call of the
// step fails in between, when the fork goes out of scope: the caller's
// stream never runs ahead of work left on the extra streams.
class Fork {
  public:
    Fork(cudaStream_t s, DeviceRes& R) : s_(s), R_(R) {}
    zero_status_t open() {
        cudaError_t e = cudaEventRecord(R_.fork, s_);
        for (int i = 0; e == cudaSuccess && i < kLanes - 1; ++i) e = cudaStreamWaitEvent(R_.aux[i], R_.fork, 0);
        open_ = e == cudaSuccess;
        return open_ ? ZERO_OK : cuda_fail("zero_step: fork", e);
    }
    zero_status_t join() {
        if (!open_) return ZERO_OK;
        open_ = false;
        for (int i = 0; i < kLanes - 1; ++i) {
            zero_status_t rc = wait_on(s_, R_.join[i], R_.aux[i], "zero_step: join");
            if (rc != ZERO_OK) return rc;
        }
        return ZERO_OK;
    }
    ~Fork() {  // after a failed call: join without replacing that call's error message
        if (!open_) return;
        for (int i = 0; i < kLanes - 1; ++i)
            if (cudaEventRecord(R_.join[i], R_.aux[i]) == cudaSuccess) cudaStreamWaitEvent(s_, R_.join[i], 0);
    }

  private:
    cudaStream_t s_;
    DeviceRes& R_;
    bool open_ = false;
};

using Ready = std::function<zero_status_t(int32_t, cudaStream_t)>;

// Mean bucket length up to which consecutive bucket launches rotate over
// several streams.  GB300, 350M layout, fused step: rotating raised every
// bucket size measured, 1e5 to 5e7 elements (5e7 at N_d = 2, 8 buckets: 6.11
// TB/s on one stream, 6.37 rotated); the 1.5B run's 500M-element buckets
// drain in about 0.1% of a launch and stay on one stream.
constexpr int64_t kAlternateMaxElems = (int64_t)1 << 27;

// The step's calls on `s`.  ready(k, stream) runs before the first call that
// reads the gradient replicas of bucket k (ZeRO-3: unit k), on the stream
// that call is issued on.
//
// Consecutive bucket launches of ZeRO-1/2 touch disjoint elements and write
// their norm partials to fixed, disjoint slots, so short ones rotate over `s`
// and the device's extra streams: the next bucket's CTAs start on the SMs
// that the previous buckets' last CTAs free, instead of after their grids
// have drained.  The extra streams join `s` before the global norm.  Results
// do not depend on the rotation: every output element and partial has one
// writer.
// Micro-batch `micro` of `n_micro` (n_micro = 1: the plain step).  Before
// the last one the step stops after its reductions; ZeRO-1 only accumulates
// locally (into `acc`) until the last one, which reduces the accumulators.
struct Micro {
    int32_t micro = 0, n_micro = 1;
    float* const* acc = nullptr;
    bool last() const { return micro == n_micro - 1; }
};

// `released`, if not null, is recorded on `s` once every launch that reads
// the gradient replicas has been issued (and joined to `s`).
zero_status_t run_step(const zero_layout* L, const zero_step_args* a, cudaStream_t s, DeviceRes& R,
                       const Ready& ready, const Micro& mb = Micro(), cudaEvent_t released = nullptr) {
    zero_status_t rc;
    auto release = [&]() -> zero_status_t {
        if (!released) return ZERO_OK;
        cudaError_t e = cudaEventRecord(released, s);
        return e == cudaSuccess ? ZERO_OK : cuda_fail("zero_step: record", e);
    };
    const int32_t nb = (int32_t)L->buckets.size();
    const zero_stream_t zs = reinterpret_cast<zero_stream_t>(s);
    // the reduction of bucket (ZeRO-3: unit) k on stream `st`
    auto reduce = [&](int32_t k, zero_stream_t st, void* const* out16, int32_t out_kind) -> zero_status_t {
        if (a->fused)
            return traced(ZERO_CALL_FUSED_STEP, reinterpret_cast<cudaStream_t>(st), [&] {
                return zero_fused_step(L, k, a->hp, a->grad_replicas, a->master, a->m, a->v, a->state, out16,
                                       out_kind, a->workspace, st);
            });
        return traced(ZERO_CALL_REDUCE_SCATTER, reinterpret_cast<cudaStream_t>(st), [&] {
            if (mb.n_micro == 1)
                return zero_reduce_scatter(L, k, a->grad_replicas, a->grad_shards, a->state, a->workspace, st);
            if (L->stage == 1)
                return zero_reduce_scatter_accumulated(L, k, (const float* const*)mb.acc, a->grad_shards,
                                                       mb.n_micro, a->state, a->workspace, st);
            return zero_reduce_scatter_micro(L, k, mb.micro, mb.n_micro, a->grad_replicas, a->grad_shards, a->state,
                                             a->workspace, st);
        });
    };
    if (L->stage == 3) {
        // One transient buffer: every unit on `s`.  Two (transient2): the
        // pages' prefetch with two live units -- consecutive units alternate
        // buffers and streams, so a unit's gather runs while the previous
        // unit's reduce-scatter and update drain.  A unit's gather and its
        // update stay on one stream (the update rewrites the 16-bit shard the
        // gather reads); units sharing a buffer share a stream; the extra
        // stream joins `s` after the forward gathers and again before the norm.
        const int32_t U = (int32_t)L->segs.size();
        const bool two = a->transient2 != nullptr && U > 1;
        auto lane = [&](int32_t i, cudaStream_t& st, void* const*& buf) {
            const bool odd = two && (i & 1);
            st = odd ? R.aux[0] : s;
            buf = odd ? a->transient2 : a->transient;
        };
        Fork fork(s, R);
        if (two && (rc = fork.open()) != ZERO_OK) return rc;
        for (int32_t u = 0; u < U; ++u) {  // forward
            cudaStream_t st;
            void* const* buf;
            lane(u, st, buf);
            const zero_stream_t zst = reinterpret_cast<zero_stream_t>(st);
            if ((rc = traced(ZERO_CALL_STAGE3_GATHER, st, [&] {
                     return zero_stage3_gather_layer(L, u, (const void* const*)a->param16_shards, buf, zst);
                 })) != ZERO_OK)
                return rc;
            if (a->unit_hook) a->unit_hook(a->hook_user, 0, u, buf, zst);
        }
        if (two) {  // forward reads of every unit end before any update rewrites a shard
            if ((rc = fork.join()) != ZERO_OK) return rc;
            if ((rc = fork.open()) != ZERO_OK) return rc;
        }
        for (int32_t u = U - 1, i = 0; u >= 0; --u, ++i) {  // backward
            cudaStream_t st;
            void* const* buf;
            lane(i, st, buf);
            const zero_stream_t zst = reinterpret_cast<zero_stream_t>(st);
            if ((rc = traced(ZERO_CALL_STAGE3_GATHER, st, [&] {
                     return zero_stage3_gather_layer(L, u, (const void* const*)a->param16_shards, buf, zst);
                 })) != ZERO_OK)
                return rc;
            if (a->unit_hook) a->unit_hook(a->hook_user, 1, u, buf, zst);
            if ((rc = ready(u, st)) != ZERO_OK) return rc;
            if ((rc = reduce(u, zst, a->param16_shards, ZERO_OUT_SHARDS)) != ZERO_OK) return rc;
        }
        if ((rc = fork.join()) != ZERO_OK) return rc;
        if ((rc = release()) != ZERO_OK) return rc;
        if (!mb.last()) return ZERO_OK;  // more micro-batches to reduce before the update
        if (a->fused)
            return traced(ZERO_CALL_GRAD_NORM, s, [&] {
                return zero_grad_norm(L, 0.0, ZERO_NORM_AFTER_FUSED, a->state, a->workspace, zs);
            });
        if ((rc = traced(ZERO_CALL_GRAD_NORM, s, [&] {
                 return zero_grad_norm(L, a->max_norm, ZERO_NORM_DECIDE, a->state, a->workspace, zs);
             })) != ZERO_OK)
            return rc;
        return traced(ZERO_CALL_ADAMW, s, [&] {
            return zero_adamw_shard_step(L, a->hp, a->master, a->m, a->v, (const float* const*)a->grad_shards,
                                         a->state, a->param16_shards, ZERO_OUT_SHARDS, zs);
        });
    }
    if (mb.n_micro > 1 && L->stage == 1) {
        // ZeRO-1 accumulates every rank's full gradient locally; only the last
        // micro-batch communicates (reading notes §4.1)
        if ((rc = traced(ZERO_CALL_ACCUMULATE, s, [&] {
                 return zero_accumulate_grads(L, mb.micro, a->grad_replicas, mb.acc, zs);
             })) != ZERO_OK)
            return rc;
        if (!mb.last()) return ZERO_OK;
    }
    const bool one_launch = a->fused && !a->per_bucket;
    if (one_launch) {
        for (int32_t b = nb - 1; b >= 0; --b)
            if ((rc = ready(b, s)) != ZERO_OK) return rc;
        if ((rc = traced(ZERO_CALL_FUSED_STEP, s, [&] {
                 return zero_fused_step(L, -1, a->hp, a->grad_replicas, a->master, a->m, a->v, a->state,
                                        a->param16_full, ZERO_OUT_FULL_REPLICAS, a->workspace, zs);
             })) != ZERO_OK)
            return rc;
        if ((rc = release()) != ZERO_OK) return rc;
    } else {
        // rotate only short buckets: a launch's ramp and drain cost a few
        // microseconds, which matters at 5M-50M elements per bucket, not at 500M
        const bool two = nb > 1 && L->psi_pad / nb <= kAlternateMaxElems;
        Fork fork(s, R);
        if (two && (rc = fork.open()) != ZERO_OK) return rc;
        for (int32_t b = nb - 1, i = 0; b >= 0; --b, ++i) {  // last bucket first
            const int lane = two ? i % kLanes : 0;
            const cudaStream_t sb = lane ? R.aux[lane - 1] : s;
            const zero_stream_t zb = reinterpret_cast<zero_stream_t>(sb);
            if ((rc = ready(b, sb)) != ZERO_OK) return rc;
            if ((rc = reduce(b, zb, a->param16_full, ZERO_OUT_FULL_REPLICAS)) != ZERO_OK) return rc;
        }
        if ((rc = fork.join()) != ZERO_OK) return rc;
        if ((rc = release()) != ZERO_OK) return rc;
        if (!mb.last()) return ZERO_OK;  // ZeRO-2: more micro-batches before the update
    }
    if (a->fused)
        return traced(ZERO_CALL_GRAD_NORM, s, [&] {
            return zero_grad_norm(L, 0.0, ZERO_NORM_AFTER_FUSED, a->state, a->workspace, zs);
        });
    if ((rc = traced(ZERO_CALL_GRAD_NORM, s, [&] {
             return zero_grad_norm(L, a->max_norm, ZERO_NORM_DECIDE, a->state, a->workspace, zs);
         })) != ZERO_OK)
        return rc;
    if (!a->param16_shards)
        return traced(ZERO_CALL_ADAMW, s, [&] {
            return zero_adamw_shard_step(L, a->hp, a->master, a->m, a->v, (const float* const*)a->grad_shards,
                                         a->state, a->param16_full, ZERO_OUT_FULL_REPLICAS, zs);
        });
    if ((rc = traced(ZERO_CALL_ADAMW, s, [&] {
             return zero_adamw_shard_step(L, a->hp, a->master, a->m, a->v, (const float* const*)a->grad_shards,
                                          a->state, a->param16_shards, ZERO_OUT_SHARDS, zs);
         })) != ZERO_OK)
        return rc;
    return traced(ZERO_CALL_ALLGATHER, s, [&] {
        return zero_allgather_params(L, (const void* const*)a->param16_shards, a->param16_full, zs);
    });
}

}  // namespace

extern "C" zero_status_t zero_step(const zero_layout* L, const zero_step_args* a, zero_stream_t stream) {
    clear_error();
    zero_status_t rc = check_args(L, a, "zero_step");
    if (rc != ZERO_OK) return rc;
    DeviceRes* R = nullptr;
    if ((rc = current_res(&R, "zero_step")) != ZERO_OK) return rc;
    std::lock_guard<std::mutex> lock(R->mu);  // the fork/join events are shared by the device's calls
    R->released_ok = false;                    // this step reads the replicas on `stream`
    if ((rc = step_res(*R, "zero_step")) != ZERO_OK) return rc;
    return run_step(L, a, reinterpret_cast<cudaStream_t>(stream), *R,
                    [](int32_t, cudaStream_t) { return ZERO_OK; });
}

extern "C" zero_status_t zero_micro_step(const zero_layout* L, const zero_step_args* a, int32_t micro,
                                         int32_t n_micro, float* const* acc_replicas, zero_stream_t stream) {
    clear_error();
    const char* what = "zero_micro_step";
    zero_status_t rc = check_args(L, a, what);
    if (rc != ZERO_OK) return rc;
    if (n_micro < 1 || micro < 0 || micro >= n_micro)
        return fail(ZERO_ERR_INVALID, "zero_micro_step: need 0 <= micro < n_micro");
    if (n_micro > 1 && a->fused)
        return fail(ZERO_ERR_INVALID, "zero_micro_step: gradient accumulation uses the split step (fused = 0)");
    if (n_micro > 1 && L->stage == 1) {
        if (!acc_replicas) return fail(ZERO_ERR_INVALID, "zero_micro_step: ZeRO-1 needs acc_replicas");
        if ((rc = check_ptrs((const void* const*)acc_replicas, L->n_d, "zero_micro_step acc_replicas")) != ZERO_OK)
            return rc;
    }
    DeviceRes* R = nullptr;
    if ((rc = current_res(&R, what)) != ZERO_OK) return rc;
    std::lock_guard<std::mutex> lock(R->mu);
    R->released_ok = false;
    if ((rc = step_res(*R, what)) != ZERO_OK) return rc;
    Micro mb;
    mb.micro = micro;
    mb.n_micro = n_micro;
    mb.acc = acc_replicas;
    return run_step(L, a, reinterpret_cast<cudaStream_t>(stream), *R,
                    [](int32_t, cudaStream_t) { return ZERO_OK; }, mb);
}

extern "C" zero_status_t zero_step_from_host(const zero_layout* L, const zero_step_args* a,
                                             const void* const* host_grads, int64_t chunk_elems,
                                             void* host_state, zero_stream_t stream) {
    clear_error();
    const char* what = "zero_step_from_host";
    zero_status_t rc = check_args(L, a, what);
    if (rc != ZERO_OK) return rc;
    if (!host_grads) return fail(ZERO_ERR_INVALID, "zero_step_from_host: NULL host gradient array");
    if (!a->grad_replicas) return fail(ZERO_ERR_INVALID, "zero_step_from_host: NULL device gradient array");
    for (int r = 0; r < L->n_d; ++r) {
        if (!host_grads[r]) return fail(ZERO_ERR_INVALID, "zero_step_from_host: NULL host gradient replica");
        if (!a->grad_replicas[r]) return fail(ZERO_ERR_INVALID, "zero_step_from_host: NULL device gradient replica");
    }
    if (chunk_elems <= 0) chunk_elems = (int64_t)1 << 27;
    DeviceRes* R = nullptr;
    if ((rc = current_res(&R, what)) != ZERO_OK) return rc;
    std::lock_guard<std::mutex> lock(R->mu);  // the events are reused by every call on this device
    const bool prev_released = R->released_ok;
    R->released_ok = false;
    if ((rc = step_res(*R, what)) != ZERO_OK) return rc;
    for (int i = 0; i < 2; ++i)
        if ((rc = make_stream(&R->cs[i], what)) != ZERO_OK) return rc;
    if ((rc = make_event(&R->start, what)) != ZERO_OK) return rc;
    if ((rc = make_event(&R->released, what)) != ZERO_OK) return rc;
    const int32_t nb = (int32_t)L->buckets.size();
    while (R->ev.size() < 2 * (size_t)nb) {
        cudaEvent_t x = nullptr;
        if ((rc = make_event(&x, what)) != ZERO_OK) return rc;
        R->ev.push_back(x);
    }
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(s, &cap)) != cudaSuccess) return cuda_fail("zero_step_from_host: capture query", e);
    const bool capturing = cap != cudaStreamCaptureStatusNone;
    // The previous step has finished reading the replicas before they are
    // overwritten: all work queued on `stream`, or, with overlap_previous,
    // the previous call's last replica-reading launch (and what came before).
    bool same = prev_released && R->released_stream == s && R->released_grads.size() == (size_t)L->n_d;
    for (int r = 0; same && r < L->n_d; ++r) same = R->released_grads[r] == a->grad_replicas[r];
    cudaEvent_t gate = R->released;
    if (!(a->overlap_previous && same && !capturing)) {
        if ((e = cudaEventRecord(R->start, s)) != cudaSuccess) return cuda_fail("zero_step_from_host: record", e);
        gate = R->start;
    }
    for (int i = 0; i < 2; ++i)
        if ((e = cudaStreamWaitEvent(R->cs[i], gate, 0)) != cudaSuccess)
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
                                    cudaMemcpyHostToDevice, R->cs[i % 2]);
                if (e != cudaSuccess) return cuda_fail("zero_step_from_host: host-to-device copy", e);
            }
        }
        for (int q = 0; q < 2; ++q)
            if ((e = cudaEventRecord(R->ev[2 * k + q], R->cs[q])) != cudaSuccess)
                return cuda_fail("zero_step_from_host: record", e);
    }
    rc = run_step(
        L, a, s, *R,
        [&](int32_t k, cudaStream_t on) -> zero_status_t {
            for (int q = 0; q < 2; ++q) {
                cudaError_t w = cudaStreamWaitEvent(on, R->ev[2 * k + q], 0);
                if (w != cudaSuccess) return cuda_fail("zero_step_from_host: wait", w);
            }
            return ZERO_OK;
        },
        Micro(), capturing ? nullptr : R->released);
    if (rc != ZERO_OK) return rc;
    if (host_state) {
        e = cudaMemcpyAsync(host_state, a->state, sizeof(zero_step_state), cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail("zero_step_from_host: state read-back", e);
    }
    R->released_stream = s;
    R->released_grads.assign(a->grad_replicas, a->grad_replicas + L->n_d);
    R->released_ok = !capturing;
    return ZERO_OK;
}

extern "C" int32_t zero_trace_enable(int32_t on) { return g_trace_on.exchange(on ? 1 : 0); }

namespace {
// Start and duration (ms) of every record, on one time axis per device: the
// offset from that device's first recorded event.  Waits for the events.
// Call with g_trace_mu held.
zero_status_t trace_times(std::vector<std::pair<float, float>>& times, const char* what) {
    times.clear();
    times.reserve(g_trace.size());
    cudaEvent_t ref[64] = {nullptr};
    for (const TraceRecord& t : g_trace) {
        cudaError_t e = cudaEventSynchronize(t.e1);
        float ms = 0.0f, at = 0.0f;
        if (!ref[t.dev]) ref[t.dev] = t.e0;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.e0, t.e1);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&at, ref[t.dev], t.e0);
        if (e != cudaSuccess) return cuda_fail(what, e);
        times.push_back({at, ms});
    }
    return ZERO_OK;
}

void trace_clear() {  // with g_trace_mu held: the events go back to the pools
    for (const TraceRecord& t : g_trace) {
        g_trace_free[t.dev].push_back(t.e0);
        g_trace_free[t.dev].push_back(t.e1);
    }
    g_trace.clear();
}
}  // namespace

extern "C" zero_status_t zero_trace_read(zero_trace_totals* out, int32_t reset) {
    clear_error();
    if (!out) return fail(ZERO_ERR_INVALID, "zero_trace_read: NULL output");
    *out = zero_trace_totals{};
    std::lock_guard<std::mutex> lock(g_trace_mu);
    std::vector<std::pair<float, float>> times;
    zero_status_t rc = trace_times(times, "zero_trace_read");
    if (rc != ZERO_OK) return rc;
    // busy time per kind: the union of its calls' intervals, placed on one
    // time axis per device by their offsets from that device's first event
    std::vector<std::pair<double, double>> spans[ZERO_CALL_KINDS];
    for (size_t i = 0; i < g_trace.size(); ++i) {
        const TraceRecord& t = g_trace[i];
        const double at = times[i].first, ms = times[i].second;
        if (t.kind >= 0 && t.kind < ZERO_CALL_KINDS) {
            out->calls[t.kind] += 1;
            out->total_ms[t.kind] += ms;
            spans[t.kind].push_back({at + 1e6 * t.dev, at + 1e6 * t.dev + ms});
        }
    }
    for (int k = 0; k < ZERO_CALL_KINDS; ++k) {
        auto& v = spans[k];
        std::sort(v.begin(), v.end());
        double busy = 0.0, lo = 0.0, hi = -1.0;
        for (const auto& p : v) {
            if (p.first > hi) {
                if (hi > lo) busy += hi - lo;
                lo = p.first;
                hi = p.second;
            } else if (p.second > hi) {
                hi = p.second;
            }
        }
        if (hi > lo) busy += hi - lo;
        out->busy_ms[k] = busy;
    }
    if (reset) trace_clear();
    return ZERO_OK;
}

extern "C" zero_status_t zero_trace_timeline(zero_trace_record* out, int64_t capacity, int64_t* count,
                                             int32_t reset) {
    clear_error();
    if (!count) return fail(ZERO_ERR_INVALID, "zero_trace_timeline: NULL count");
    if (capacity < 0 || (capacity > 0 && !out))
        return fail(ZERO_ERR_INVALID, "zero_trace_timeline: need capacity >= 0 and an output array");
    std::lock_guard<std::mutex> lock(g_trace_mu);
    std::vector<std::pair<float, float>> times;
    zero_status_t rc = trace_times(times, "zero_trace_timeline");
    if (rc != ZERO_OK) return rc;
    *count = (int64_t)g_trace.size();
    const size_t n = std::min((size_t)capacity, g_trace.size());
    for (size_t i = 0; i < n; ++i) {
        const TraceRecord& t = g_trace[i];
        out[i].kind = t.kind;
        out[i].device = t.dev;
        out[i].stream = (uint64_t)(uintptr_t)t.stream;
        out[i].start_ms = times[i].first;
        out[i].end_ms = (double)times[i].first + times[i].second;
    }
    if (reset) trace_clear();
    return ZERO_OK;
}
