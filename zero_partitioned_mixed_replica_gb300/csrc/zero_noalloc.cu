// Allocation-free whole fused step.
//
// Some callers cannot hand the library a device workspace: a plug-in running
// inside a host application that owns every byte of device memory through its
// own pool, or a latency-critical loop that must never call cudaMalloc because
// the call can synchronise the device.  For them, zero_fused_step_noalloc runs
// the same fused step as zero_fused_step + zero_grad_norm(AFTER_FUSED), but
// keeps the norm scratch (one float per 32 parameters plus the 1024 block sums)
// in the file-scope device array below instead of a caller workspace.
//
// The array is part of the library image: every GPU that loads libzero.so
// holds these 8 MiB + 8 KiB until the process exits.  All calls share it and
// it keeps the last call's contents; nothing needs clearing, because every slot
// a call reads is written earlier in the same call.  Calls that overlap on the
// GPU (several streams, or several host threads) race on the array.
#include <cstddef>
#include <mutex>

#include "zero_launch.h"

namespace {

constexpr int64_t kNoallocMaxElems = ZERO_NOALLOC_MAX_ELEMS;
constexpr size_t kPartialBytes = (size_t)(kNoallocMaxElems / zero_detail::kGroup) * sizeof(float);
constexpr size_t kScratchBytes = kPartialBytes + (size_t)zero_detail::kNormBlocks * sizeof(double);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Unique id of the calling thread's current CUDA context, through the
// driver's cuCtxGetCurrent / cuCtxGetId reached by the runtime's entry-point
// query (the library links no driver library).  False if there is no current
// context yet or the query is unavailable.
bool current_context_id(unsigned long long* id) {
    typedef int (*get_current_fn)(void**);
    typedef int (*get_id_fn)(void*, unsigned long long*);
    static get_current_fn get_current = nullptr;
    static get_id_fn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<get_current_fn>(f);
        f = nullptr;
        q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<get_id_fn>(f);
    });
    if (!get_current || !get_id) return false;
    void* ctx = nullptr;
    if (get_current(&ctx) != 0 || !ctx) return false;
    return get_id(ctx, id) == 0;
}

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol names a host-side stand-in, so the address is looked up with the
// device current, at the first call on that device, and cached together with
// the id of the context it belongs to.  A call under another context of the
// same device (after cudaDeviceReset, or after the primary context was
// released and created again) looks the address up again instead of using a
// stale one.
zero_status_t scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    static unsigned long long ctx_of[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return zero_detail::fail(ZERO_ERR_CUDA, std::string("zero_fused_step_noalloc: ") +
                                                                      cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return zero_detail::fail(ZERO_ERR_CUDA, "zero_fused_step_noalloc: device index >= 64");
    std::lock_guard<std::mutex> lock(mu);
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    if (!addr[dev] || !have_id || id != ctx_of[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return zero_detail::fail(ZERO_ERR_CUDA, std::string("zero_fused_step_noalloc: cudaGetSymbolAddress: ") +
                                                        cudaGetErrorString(e));
        addr[dev] = p;
        // the lookup makes the device's primary context current if none was
        ctx_of[dev] = current_context_id(&id) ? id : 0;
    }
    *out = addr[dev];
    return ZERO_OK;
}

}  // namespace

using namespace zero_detail;

extern "C" zero_status_t zero_fused_step_noalloc(const zero_layout* L, const zero_adamw_hp* hp,
                                                 const void* const* grad_replicas, float* const* master,
                                                 float* const* m, float* const* v, zero_step_state* st,
                                                 void* const* param16_out, int32_t out_kind,
                                                 zero_stream_t stream) {
    clear_error();
    if (!L) return fail(ZERO_ERR_INVALID, "zero_fused_step_noalloc: NULL layout");
    if (L->stage == 0) return fail(ZERO_ERR_STATE, "zero_fused_step_noalloc: stage 0 has no partitioned step");
    if (L->psi_pad > kNoallocMaxElems || workspace_bytes(L) > (int64_t)kScratchBytes)
        return fail(ZERO_ERR_INVALID,
                    "zero_fused_step_noalloc: Psi_pad " + std::to_string(L->psi_pad) +
                        " exceeds the built-in scratch limit of " + std::to_string(kNoallocMaxElems) +
                        " padded elements; use zero_fused_step with a caller workspace");
    void* scratch = nullptr;
    zero_status_t rc = scratch_address(&scratch);
    if (rc != ZERO_OK) return rc;
    if (L->stage == 3) {
        for (int32_t u = (int32_t)L->segs.size() - 1; u >= 0; --u) {
            rc = zero_fused_step(L, u, hp, grad_replicas, master, m, v, st, param16_out, out_kind, scratch, stream);
            if (rc != ZERO_OK) return rc;
        }
    } else {
        rc = zero_fused_step(L, -1, hp, grad_replicas, master, m, v, st, param16_out, out_kind, scratch, stream);
        if (rc != ZERO_OK) return rc;
    }
    return zero_grad_norm(L, 0.0, ZERO_NORM_AFTER_FUSED, st, scratch, stream);
}
