/*
 * zero.h — C ABI of libzero: the ZeRO-DP partitioned mixed-precision AdamW
 * step on one GB300 (sm_103a), with N_d simulated data-parallel ranks held as
 * separate device buffers.
 *
 * One step (ZeRO-1/2): reduce-scatter the N_d 16-bit gradient replicas over a
 * flat, padded, bucketed parameter buffer; compute the global gradient norm
 * from every rank's partial sums; apply AdamW to each rank's fp32
 * master/m/v shard; cast to 16 bits and all-gather into every rank's full
 * parameter replica.  ZeRO-3 instead gathers the 16-bit shards of one unit
 * (a transformer block, or the root unit with embeddings and head) into a
 * transient buffer before forward and again before backward, reduce-scatters
 * per unit and writes only the rank's 16-bit shard (no all-gather at the end
 * of the step).
 *
 * Sources, by page title and section:
 *   [L5]  "第 5 课：ZeRO 与 FSDP" (hsthanb4.github.io, hpclearning lesson 5):
 *         §2 memory formulas, §3 reduce-scatter / update / all-gather and the
 *         2Psi vs 3Psi volumes, Fig. 5-1 per-layer gather-and-release.
 *   [RN]  "ZeRO: Memory Optimizations Toward Training Trillion Parameter
 *         Models" (reading notes, unpurerationalist.github.io): §2.1 mixed
 *         precision (fp32 master, m, v), §2.2 fp32 fused buffers, §3.1 dynamic
 *         communication schedule, §4.1-§4.3 P_os / P_g / P_p, §5.2 constant
 *         size buffers, §6 communication volumes.
 *   [Z3]  "ZeRO-3 核心流程：把参数也切开的那一档" (llmnex.top): §2 the four actions
 *         per layer, 坑 1 sharding-aware gradient clipping.
 *   [FS]  "別再複製本可分片的東西：ZeRO 與 FSDP" (jovanaeducation.com): FSDP units.
 *   [ML]  mlqm.cn data-parallel / ZeRO post: gradient buckets, ds_config.
 * Where the pages are silent (AdamW formula, padding, bucket boundaries,
 * rounding, loss scaling, overflow skip) the readings are stated at the
 * function that uses them.
 *
 * Conventions for every call:
 *   - Ownership: the caller allocates and owns every device buffer (master,
 *     m, v, replicas, shards, transients, workspace, state).  The library
 *     never allocates device memory and never frees a caller pointer.  Only
 *     the zero_layout object is library-owned (zero_layout_destroy frees it).
 *   - Pointer arrays (`... const* x`) are HOST arrays of N_d DEVICE pointers,
 *     one per simulated rank, read during the call only.
 *   - Alignment: every device buffer must start on a 256-byte boundary, else
 *     ZERO_ERR_ALIGN.  NULL where a buffer is required: ZERO_ERR_INVALID.
 *   - Asynchrony: device calls enqueue kernels on `stream` and return without
 *     synchronising the host.  A launch error returns ZERO_ERR_CUDA; a fault
 *     during execution surfaces at the caller's next synchronisation.
 *   - Status: no exception or abort crosses the ABI; the return value is the
 *     only channel.  zero_last_error() gives a message for the last failing
 *     call on the calling thread.
 *   - Layout constants: q = N_d * 128 (or pad_multiple); Psi_pad = padded
 *     flat length; S = per-rank shard length.  Rank r owns flat range
 *     [r*S, (r+1)*S) for ZeRO-1/2, and slice [r*S_u, (r+1)*S_u) of every unit u
 *     for ZeRO-3 (its shard is those slices concatenated in unit order).
 */
#ifndef ZERO_H
#define ZERO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-compatible with cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st* zero_stream_t;

typedef int32_t zero_status_t;
enum {
    ZERO_OK = 0,
    ZERO_ERR_INVALID = -1, /* bad argument, size, index, stage or NULL pointer */
    ZERO_ERR_ALIGN = -2,   /* a device buffer is not 256-byte aligned        */
    ZERO_ERR_CUDA = -3,    /* a CUDA launch or query failed                  */
    ZERO_ERR_STATE = -4,   /* call not valid for this layout's stage          */
    ZERO_ERR_TIMEOUT = -5, /* reserved: no host call waits on the device      */
    ZERO_ERR_NOMEM = -6    /* host allocation of the layout object failed     */
};

typedef enum { ZERO_BF16 = 0, ZERO_FP16 = 1 } zero_dtype_t;

#define ZERO_MAX_RANKS 64

/* Output kinds of zero_adamw_shard_step / zero_fused_step. */
enum {
    ZERO_OUT_FULL_REPLICAS = 0, /* ZeRO-1/2: write each updated 16-bit value into
                                   all N_d full replicas (all-gather fused)     */
    ZERO_OUT_SHARDS = 1         /* write rank r's 16-bit shard only (ZeRO-3, or
                                   ZeRO-1/2 followed by zero_allgather_params)  */
};

/* Flags of zero_grad_norm. */
enum {
    ZERO_NORM_DECIDE = 0,      /* split step: decide skip/clip before the update */
    ZERO_NORM_AFTER_FUSED = 1  /* fused step: the update already ran; record the
                                  norm and advance the step counter            */
};

typedef struct zero_layout zero_layout; /* opaque, immutable after init */

/* Everything zero_layout_query reports.  Bytes are per rank; counters are
 * elements moved per rank per step. */
typedef struct zero_layout_info {
    int32_t n_d, stage, dtype, n_tensors;
    int32_t n_buckets, n_units, reserved0, reserved1;
    int64_t psi;             /* real parameter count                          */
    int64_t psi_pad;         /* padded flat length                            */
    int64_t q;               /* padding quantum                               */
    int64_t bucket_elems;    /* requested bucket size (<= 0: one bucket)      */
    int64_t shard_len;       /* S: per-rank shard length (sum of S_u)         */
    int64_t max_unit_padded; /* largest padded segment                        */
    /* memory per rank, [L5] §2 M0..M3 with Psi -> Psi_pad and Psi/N_d -> S */
    int64_t mem_formula;     /* M_stage                                       */
    int64_t mem_state;       /* fp32 master + m + v shard: 12 S               */
    int64_t mem_gshard;      /* fp32 reduced-gradient shard: 4 S ([RN] §2.2)   */
    int64_t mem_transient;   /* ZeRO-3: 2 bytes x largest padded unit, else 0  */
    int64_t mem_peak;        /* mem_formula + mem_transient                   */
    /* communication per rank, [L5] §3 / [RN] §6: (N_d - 1) * S per collective */
    int64_t comm_rs, comm_ag, comm_ag_fwd, comm_ag_bwd, comm_allreduce, comm_total;
    int64_t workspace_bytes; /* device workspace the step calls need          */
} zero_layout_info;

/* One separately padded segment: the whole buffer for ZeRO-0/1/2, a unit for
 * ZeRO-3. */
typedef struct zero_unit_info {
    int64_t offset;     /* flat offset                                        */
    int64_t real;       /* real element count                                 */
    int64_t padded;     /* padded element count (multiple of q)              */
    int64_t shard;      /* S_u = padded / N_d                                 */
    int64_t shard_base; /* offset of this segment inside every rank's shard  */
} zero_unit_info;

/* Device-resident step state (96 bytes).  Create it with zero_state_init;
 * only the library's kernels write it afterwards.  The host may read it
 * (after synchronising) to see the norm, the overflow flag and the counters. */
typedef struct zero_step_state {
    double beta1, beta2;         /* AdamW betas                                 */
    double beta1_pow, beta2_pow; /* beta^t after t applied steps (t products)   */
    double grad_norm;            /* global norm of the last step (+inf: overflow) */
    float loss_scale;            /* current loss scale                          */
    float clip_coef;             /* clip coefficient of the last step (1: none) */
    int32_t t;                   /* applied (not skipped) steps                 */
    int32_t skipped;             /* skipped steps                               */
    int32_t good_steps;          /* applied steps since the last scale change   */
    int32_t growth_interval;     /* double the scale after this many good steps */
    int32_t dynamic_scale;       /* 1: halve on overflow, grow after interval   */
    int32_t nonfinite;           /* OR of this step's reduce-scatter checks     */
    int32_t overflow;            /* last decided step overflowed                */
    int32_t apply;               /* last decided step applies the update        */
    int32_t error;               /* device-detected errors, OR of bits (0 = none):
                                    1 = a bounded wait of a kernel on its own bulk
                                    copies ran out; that CTA drained its copies and
                                    stopped, so the step's results are incomplete;
                                    2 = also, while draining, one of those copies
                                    did not land within 4 more bounded waits: the
                                    CTA exited with it possibly still in flight,
                                    so treat the context as unreliable */
    int32_t reserved[3];
} zero_step_state;

/* AdamW hyperparameters that may change between steps (lr schedules).  The
 * betas live in zero_step_state.  lr >= 0, weight_decay >= 0, eps > 0 also
 * once rounded to binary32 (eps > 2^-150); anything else is ZERO_ERR_INVALID. */
typedef struct zero_adamw_hp {
    double lr;
    double eps;
    double weight_decay;
} zero_adamw_hp;

/* ------------------------------------------------------------------------ */
/* Layout (host only, integer work)                                          */
/* ------------------------------------------------------------------------ */

/* Flatten, pad, shard, bucket and account ([RN] §2.2 and §5.2 flatten into one
 * contiguous buffer; [L5] §2 and [RN] §4 equal 1/N_d split; [ML] "梯度桶化" and
 * [RN] §4.1-§4.2 fixed-size buckets; [FS] one unit per block plus a root unit).
 *   numels[n_tensors]   element count of each tensor, declaration order (> 0).
 *   unit_of_tensor      ZeRO-3 unit id per tensor (0..U-1, none empty), or
 *                       NULL for stages 0-2 (required for stage 3).
 *   n_d                 simulated ranks, 1..ZERO_MAX_RANKS.
 *   stage               0 (DDP: accounting only), 1, 2 or 3.
 *   pad_multiple        0 => q = n_d*128; else a positive multiple of n_d*128.
 *   bucket_elems        <= 0: one bucket; else a multiple of 32.  Buckets are
 *                       [k*B, min((k+1)*B, Psi_pad)); ZeRO-3 buckets are units.
 *   dtype               16-bit format of gradients and parameters.
 * Readings: stages 0-2 flatten in declaration order with no gaps and pad the
 * tail with zeros to a multiple of q; stage 3 lays units out in id order, each
 * unit's tensors in declaration order, each unit padded to a multiple of q.
 * On success *out owns a new layout; on error *out is untouched. */
zero_status_t zero_layout_init(const int64_t* numels, int32_t n_tensors,
                               const int32_t* unit_of_tensor, int32_t n_d, int32_t stage,
                               int64_t pad_multiple, int64_t bucket_elems,
                               zero_dtype_t dtype, zero_layout** out);
zero_status_t zero_layout_query(const zero_layout* L, zero_layout_info* out);
/* [begin, end) of bucket b (ZeRO-3: of unit b). */
zero_status_t zero_layout_bucket(const zero_layout* L, int32_t b, int64_t* begin, int64_t* end);
zero_status_t zero_layout_unit(const zero_layout* L, int32_t u, zero_unit_info* out);
/* Flat offset of tensor t. */
zero_status_t zero_layout_tensor_offset(const zero_layout* L, int32_t t, int64_t* offset);
void zero_layout_destroy(zero_layout* L);

/* One contiguous copy of the reshard plan: len elements from rank src_rank's
 * shard at src_off to rank dst_rank's shard at dst_off. */
typedef struct zero_copy_segment {
    int32_t src_rank, dst_rank;
    int64_t src_off, dst_off, len;
} zero_copy_segment;

/* Resharding plan between two layouts of the same tensors (sharded
 * checkpoints: each rank saves its own shard, "別再複製本可分片的東西：ZeRO 與
 * FSDP", 分片檢查點; loading into another N_d, stage or unit split needs every
 * real element's new home).  Host only, integer work.  Every real element of
 * every tensor appears in exactly one segment; padding in neither.  Segments
 * are maximal (contiguous in both shard spaces), in src flat order.
 *   src, dst   layouts with equal tensor counts and sizes (any n_d, stage 1-3).
 *   out        capacity segments, or NULL to query the count.
 *   *count     number of segments the plan needs.
 * Returns ZERO_ERR_INVALID if the tensors differ, a layout is stage 0, or
 * capacity is too small (with *count set). */
zero_status_t zero_reshard_plan(const zero_layout* src, const zero_layout* dst, zero_copy_segment* out,
                                int64_t capacity, int64_t* count);

/* ------------------------------------------------------------------------ */
/* Step state                                                                */
/* ------------------------------------------------------------------------ */

/* Write the initial state into device memory `st` (t = 0, betas, beta^0 = 1,
 * loss_scale >= 1, no error).  growth_interval >= 1.  One tiny kernel. */
zero_status_t zero_state_init(zero_step_state* st, double beta1, double beta2,
                              float loss_scale, int32_t dynamic_scale,
                              int32_t growth_interval, zero_stream_t stream);

/* ------------------------------------------------------------------------ */
/* The step                                                                  */
/* ------------------------------------------------------------------------ */

/* Reduce-scatter of one bucket (ZeRO-1/2) or one unit (ZeRO-3) ([L5] §3 step
 * 1; [RN] §4.1-§4.3 bucketed, asynchronous reduce-scatter; [Z3] §2 backward).
 * For every flat index i of the bucket, owned by rank r at shard offset j:
 *   s = x_0 + x_1 + ... + x_{N_d-1}   (x_k = grad_replicas[k][i], binary32
 *                                      adds in rank order; padding reads 0)
 *   grad_shards[r][j] = s / (N_d * loss_scale)   (IEEE division)
 * It also writes the 32-element sums of squares used by zero_grad_norm into
 * `workspace` and ORs "some s is inf/NaN" into st->nonfinite.
 *   grad_replicas: N_d device pointers to full 16-bit replicas (Psi_pad each).
 *   grad_shards:   N_d device pointers to fp32 shards (S each).
 *   workspace:     >= info.workspace_bytes, shared by all calls of a step.
 * Every bucket (unit) must be reduced once per step before zero_grad_norm.
 * Stage 0: ZERO_ERR_STATE. */
zero_status_t zero_reduce_scatter(const zero_layout* L, int32_t bucket_or_unit,
                                  const void* const* grad_replicas, float* const* grad_shards,
                                  zero_step_state* st, void* workspace, zero_stream_t stream);

/* Sharding-aware global gradient norm and the step decision ([Z3] 坑 1: the
 * norm must combine every shard's partial sums, else each rank clips by a
 * different coefficient).  Two deterministic passes over the 32-element
 * partials (binary64 from there on): norm = sqrt(sum g^2) over all Psi_pad.
 * ZERO_NORM_DECIDE (split step, before zero_adamw_shard_step):
 *   overflow = st->nonfinite.  If overflow: grad_norm = +inf, the update is
 *   skipped (apply = 0), skipped += 1, a dynamic scale halves (never below 1).
 *   Else: clip_coef = min(1, max_norm / (norm + 1e-6)) (1 if max_norm <= 0),
 *   t += 1, beta^t advance, apply = 1, and a dynamic scale doubles after
 *   growth_interval consecutive applied steps.
 * ZERO_NORM_AFTER_FUSED (after zero_fused_step): records the norm and the
 *   overflow flag, and advances t and beta^t (the update already ran).
 * Both clear st->nonfinite for the next step.  Readings: the skip rule, the
 * 1e-6 and the scale schedule are not on the pages (mixed-precision practice). */
zero_status_t zero_grad_norm(const zero_layout* L, double max_norm, int32_t flags,
                             zero_step_state* st, void* workspace, zero_stream_t stream);

/* Sharded AdamW, cast and (optionally fused) all-gather ([L5] §3 step 2: each
 * rank updates its 1/N_d fp32 state and casts it to 16 bits in place; [RN]
 * §4.1 then all-gathers; [Z3] §2 step 3 zero communication).  No-op when
 * st->apply == 0.  Per element of every rank's shard, one binary32 rounding
 * per operation, no fused multiply-add (reading: decoupled weight decay):
 *   g'  = g * clip_coef
 *   p1  = p * (1 - lr*wd)
 *   m   = beta1*m + (1-beta1)*g'
 *   v   = beta2*v + (1-beta2)*(g'*g')
 *   den = sqrt(v) / sqrt(1 - beta2^t) + eps
 *   p   = p1 - (lr / (1 - beta1^t)) * (m / den)
 *   out = round-to-nearest-even 16-bit(p)
 * Constants are computed in binary64 and rounded once to binary32.
 *   master, m, v:  N_d device pointers to fp32 shards (S each), updated in place.
 *   grad_shards:   N_d fp32 shards written by zero_reduce_scatter.
 *   param16_out:   ZERO_OUT_FULL_REPLICAS: N_d full 16-bit replicas (Psi_pad);
 *                  ZERO_OUT_SHARDS: N_d 16-bit shards (S).  ZeRO-3 requires
 *                  ZERO_OUT_SHARDS. */
zero_status_t zero_adamw_shard_step(const zero_layout* L, const zero_adamw_hp* hp,
                                    float* const* master, float* const* m, float* const* v,
                                    const float* const* grad_shards, zero_step_state* st,
                                    void* const* param16_out, int32_t out_kind,
                                    zero_stream_t stream);

/* Unfused all-gather of 16-bit shards into every rank's full replica
 * (ZeRO-1/2; [L5] §3 step 3, [RN] §6.2.1): param16_full[k][r*S + j] =
 * param16_shards[r][j] for every k, r, j.  Stage 3: ZERO_ERR_STATE. */
zero_status_t zero_allgather_params(const zero_layout* L, const void* const* param16_shards,
                                    void* const* param16_full, zero_stream_t stream);

/* The 16-bit parameters of the current fp32 master, without an update:
 * the cast of [L5] §3 step 2 ("cast the fp32 shard to BF16 in place") and,
 * for ZERO_OUT_FULL_REPLICAS, the all-gather of step 3.  For initialising
 * the 16-bit parameters from a loaded master (and after a checkpoint load).
 *   master:       N_d device pointers to fp32 shards (S each), read only.
 *   param16_out:  ZERO_OUT_FULL_REPLICAS (ZeRO-1/2): N_d full replicas
 *                 (Psi_pad each); element r*S + j of every replica receives
 *                 round-to-nearest-even 16-bit(master[r][j]).
 *                 ZERO_OUT_SHARDS: N_d 16-bit shards (S each); shard r
 *                 receives the cast of master[r].  ZeRO-3 requires it.
 * Padding casts its zeros to +0.  One kernel; asynchronous on `stream`.
 * Errors: NULL/misaligned pointers, unknown out_kind (ZERO_ERR_INVALID /
 * ZERO_ERR_ALIGN); stage 0, or ZeRO-3 with full replicas (ZERO_ERR_STATE). */
zero_status_t zero_cast_params(const zero_layout* L, const float* const* master,
                               void* const* param16_out, int32_t out_kind, zero_stream_t stream);

/* ZeRO-3 gather of unit `unit` into every rank's transient buffer ([L5]
 * Fig. 5-1; [RN] §3.1 and §4.3; [Z3] §2 steps 1-2): transient[k][i] =
 * param16_shards[r][S_u_base + i - r*S_u] for i in [0, real_u), r = i / S_u,
 * for every rank k.  The unit's padding is not written.  "Release" is the
 * caller reusing the buffer for the next unit.  transient: N_d device
 * pointers, each >= real_u 16-bit elements.  Stages 0-2: ZERO_ERR_STATE. */
zero_status_t zero_stage3_gather_layer(const zero_layout* L, int32_t unit,
                                       const void* const* param16_shards, void* const* transient,
                                       zero_stream_t stream);

/* Reduce-scatter + AdamW + cast (+ all-gather) in one pass, for steps with
 * neither clipping nor a loss scaler (the update cannot wait for a global
 * norm): the arithmetic of zero_reduce_scatter and zero_adamw_shard_step per
 * element, with clip_coef = 1 and the constants of step t + 1.  It also writes
 * the norm partials and ORs st->nonfinite; follow it (after all buckets or
 * units of the step) with zero_grad_norm(..., ZERO_NORM_AFTER_FUSED, ...).
 * bucket_or_unit: a bucket (ZeRO-1/2) or unit (ZeRO-3) index, or -1 for the
 * whole buffer.  Stage 1/2 with ZERO_OUT_FULL_REPLICAS or ZERO_OUT_SHARDS;
 * stage 3 with ZERO_OUT_SHARDS.  A non-finite gradient is reported but not
 * skipped (use the split calls when a loss scaler is active). */
zero_status_t zero_fused_step(const zero_layout* L, int32_t bucket_or_unit,
                              const zero_adamw_hp* hp, const void* const* grad_replicas,
                              float* const* master, float* const* m, float* const* v,
                              zero_step_state* st, void* const* param16_out, int32_t out_kind,
                              void* workspace, zero_stream_t stream);

/* ------------------------------------------------------------------------ */
/* The whole step in one call                                                */
/* ------------------------------------------------------------------------ */
/* Called by the step executor on the calling thread right after it has
 * issued the gather of ZeRO-3 unit `unit` on `stream` (pass 0: forward, 1:
 * backward), before it issues anything else for that unit: the place where a
 * layer's forward or backward computation on the gathered unit would be
 * enqueued.  `transient` holds the N_d buffers that gather writes.  With
 * transient2, consecutive units' hooks get different streams: work that
 * depends on the previous unit's (a layer's input is the previous layer's
 * output) must be ordered by the caller, e.g. with an event.  The hook must
 * not call zero_step, zero_micro_step or zero_step_from_host (the executor
 * holds its per-device lock). */
typedef void (*zero_unit_hook_fn)(void* user, int32_t pass, int32_t unit, void* const* transient,
                                  zero_stream_t stream);

/* Buffers and settings of one step, for zero_step and zero_step_from_host.
 * Every pointer array holds N_d device pointers (256-byte aligned); the
 * library reads the arrays during the call only. */
typedef struct zero_step_args {
    const zero_adamw_hp* hp;            /* host pointer, read during the call */
    double max_norm;                    /* split step: clip threshold (<= 0: no clip) */
    int32_t fused;                      /* 1: zero_fused_step per bucket/unit + norm report
                                           (no clip, no loss-scale skip); 0: split step */
    int32_t per_bucket;                 /* fused ZeRO-1/2: 1 = one launch per bucket,
                                           0 = one launch over the whole buffer */
    const void* const* grad_replicas;   /* 16-bit, Psi_pad each (zero_step_from_host:
                                           the device destinations of the copies) */
    float* const* master;               /* fp32 shards, S each */
    float* const* m;
    float* const* v;
    float* const* grad_shards;          /* split step: fp32 shards (S); fused: unused */
    void* const* param16_full;          /* ZeRO-1/2: full 16-bit replicas; ZeRO-3: unused */
    void* const* param16_shards;        /* ZeRO-3: 16-bit shards (S).  ZeRO-1/2 split step:
                                           NULL = the update writes param16_full directly
                                           (all-gather fused), else it writes these shards
                                           and zero_allgather_params follows */
    void* const* transient;             /* ZeRO-3: transient unit buffers (largest unit) */
    zero_step_state* state;             /* device */
    void* workspace;                    /* device, zero_layout_info.workspace_bytes */
    void* const* transient2;            /* ZeRO-3, optional: a second set of transient
                                           buffers.  Consecutive units then alternate
                                           buffers and streams (two live units, [L5]
                                           §4 prefetch): a unit's gather overlaps the
                                           previous unit's reduce-scatter and update.
                                           NULL: one buffer, one stream */
    zero_unit_hook_fn unit_hook;        /* ZeRO-3, optional: see zero_unit_hook_fn */
    void* hook_user;                    /* passed to unit_hook */
    int32_t overlap_previous;           /* zero_step_from_host only, 0 or 1: see there */
} zero_step_args;

/* One whole step with the gradient replicas resident in device memory, in the
 * pages' call order ([ML] "梯度桶化"; [RN] §4.1-§4.3; [L5] §3 and Fig. 5-1;
 * [Z3] §2):
 *   ZeRO-1/2 split: zero_reduce_scatter for every bucket, last bucket first
 *     -> zero_grad_norm(max_norm, DECIDE) -> zero_adamw_shard_step (full
 *     replicas, or shards + zero_allgather_params);
 *   ZeRO-1/2 fused: zero_fused_step per bucket, last first (or once over the
 *     buffer) -> zero_grad_norm(AFTER_FUSED);
 *   ZeRO-3: zero_stage3_gather_layer for units 0..U-1 (forward), then for
 *     u = U-1..0: gather u again and zero_fused_step(u) (fused) or
 *     zero_reduce_scatter(u) (split, followed by the norm and the shard
 *     update after the loop).  With transient2, units alternate between the
 *     two buffer sets and between `stream` and one of the library's streams;
 *     every forward gather ends before the first update.
 * ZeRO-1/2 bucket launches of short buckets (mean at most 2^27 elements)
 * rotate over `stream` and seven streams of the library's (created per device
 * at the first call), which join `stream` again before the norm: consecutive
 * buckets touch disjoint elements and norm-partial slots, so one bucket's
 * launch can start while the previous one drains.  Results do not depend on
 * it.
 * Asynchronous on `stream`; allocates no device memory; captures into a CUDA
 * graph like the calls it issues.  Calls on one device are serialised by a
 * library lock.  Errors: those of the calls it issues (the first failing call
 * stops the step and its status is returned); inconsistent arguments (fused
 * with max_norm > 0, missing buffers for the stage) give ZERO_ERR_INVALID
 * before any launch. */
zero_status_t zero_step(const zero_layout* L, const zero_step_args* args, zero_stream_t stream);

/* zero_step with the N_d gradient replicas in host memory.  host_grads: N_d
 * host pointers, Psi_pad 16-bit elements each (page-locked memory lets the
 * copies overlap the step; pageable memory is correct but copies in stages).
 * Each bucket's range (ZeRO-3: each unit's) of every replica is copied into
 * args->grad_replicas by cudaMemcpyAsync, chunk_elems elements at a time
 * (<= 0: 2^27), alternating over two copy streams that the library owns (one
 * pair per device, created at the first call and kept until exit), in the
 * order the step consumes the buckets; the step's first reading launch of
 * each bucket waits only for that bucket's copies, so later buckets cross the
 * host link while earlier ones are reduced ([RN] §4.1-§4.2: a bucket is
 * reduced as soon as it is filled).  The copies start after the work already
 * queued on `stream` (the previous step reads the same device replicas),
 * except with args->overlap_previous = 1: when the previous executor call on
 * this device was a zero_step_from_host call on the same `stream` with the
 * same device replicas (args->grad_replicas) that succeeded outside a graph
 * capture, the copies then wait only for that call's last launch that reads
 * the device replicas (its reduce-scatters or fused updates, and everything
 * queued before them), so its norm and update overlap this step's copies.
 * The caller must then queue nothing between the two calls that reads or
 * writes the device replicas: they are the library's staging buffers.  Any
 * zero_step or zero_micro_step call in between, another stream or other
 * device replicas than the previous call's, a capturing `stream`, or a failed
 * previous call makes the copies wait for all work queued on `stream`.
 * host_state: host pointer to sizeof(zero_step_state) bytes, or NULL; the
 * step state is copied there at the end of the step, on `stream`.
 * Asynchronous: synchronise `stream` before reading host_state or reusing
 * host_grads.  Calls on one device are serialised by a library lock (they
 * share the copy streams and events). */
zero_status_t zero_step_from_host(const zero_layout* L, const zero_step_args* args,
                                  const void* const* host_grads, int64_t chunk_elems, void* host_state,
                                  zero_stream_t stream);

/* Launch tracing of zero_step, zero_micro_step and zero_step_from_host.  With tracing on,
 * every library call the executor issues is bracketed by two timing events
 * recorded on the stream the call is issued on (none while that stream is
 * being captured into a CUDA graph); zero_trace_read waits for the recorded
 * events and adds up the elapsed time per kind of call.  Records accumulate
 * until a read with reset; beyond 2^20 of them, calls run untraced. */
enum {
    ZERO_CALL_REDUCE_SCATTER = 0,
    ZERO_CALL_GRAD_NORM = 1,      /* both passes of zero_grad_norm */
    ZERO_CALL_ADAMW = 2,
    ZERO_CALL_FUSED_STEP = 3,
    ZERO_CALL_STAGE3_GATHER = 4,
    ZERO_CALL_ALLGATHER = 5,
    ZERO_CALL_ACCUMULATE = 6,
    ZERO_CALL_KINDS = 7
};
typedef struct zero_trace_totals {
    int64_t calls[8];             /* traced calls per ZERO_CALL_* kind          */
    double total_ms[8];           /* sum of their event-timed durations (ms)    */
    double busy_ms[8];            /* time with at least one of them in flight:
                                     equals total_ms unless calls of the kind
                                     overlapped (alternating bucket streams)   */
} zero_trace_totals;

/* Turn tracing on (1) or off (0), process-wide; returns the previous setting. */
int32_t zero_trace_enable(int32_t on);

/* Totals of the calls traced since the last reset.  Blocks until every
 * recorded event has completed.  reset != 0 clears the record afterwards (its
 * events are reused).  Errors: NULL out (ZERO_ERR_INVALID); a failing event
 * query (ZERO_ERR_CUDA). */
zero_status_t zero_trace_read(zero_trace_totals* out, int32_t reset);

/* One traced call on a time axis (a timeline, for launch gaps and overlap
 * between streams). */
typedef struct zero_trace_record {
    int32_t kind;                 /* ZERO_CALL_*                                 */
    int32_t device;               /* CUDA device index                           */
    uint64_t stream;              /* the launching stream's handle, as an id     */
    double start_ms;              /* its first timing event, from the device's
                                     first traced event (CUDA event resolution,
                                     about 0.5 us)                              */
    double end_ms;                /* its second timing event                     */
} zero_trace_record;

/* The calls traced since the last reset, in issue order.  Blocks until every
 * recorded event has completed.  Writes min(capacity, count) records to out
 * (out may be NULL when capacity is 0, to ask for the count) and sets *count
 * to the number of records held.  reset != 0 clears the record afterwards,
 * as zero_trace_read does.  Errors: NULL count, capacity < 0, or capacity > 0
 * with a NULL out (ZERO_ERR_INVALID); a failing event query (ZERO_ERR_CUDA). */
zero_status_t zero_trace_timeline(zero_trace_record* out, int64_t capacity, int64_t* count, int32_t reset);

/* ------------------------------------------------------------------------ */
/* Gradient accumulation over M micro-batches per optimizer step             */
/* ------------------------------------------------------------------------ */
/* Reading notes "ZeRO: Memory Optimizations ..." §4.1: with P_os (ZeRO-1)
 * gradient accumulation needs no extra communication — every rank keeps its
 * full gradient and accumulates locally; §4.2 (ZeRO-2) and §4.3 (ZeRO-3)
 * reduce-scatter every micro-batch.  "第 5 课：ZeRO 与 FSDP" §2: fp32
 * accumulation costs 4 Psi per rank for ZeRO-1 and 4 Psi / N_d for ZeRO-2/3.
 * The averaged gradient is g = (sum over micro-batches and ranks) /
 * (N_d * M * loss_scale); the two schedules sum in different orders:
 *   ZeRO-1:   A_r = x_{r,0} + x_{r,1} + ...  then  g = (A_0 + A_1 + ...) / D
 *   ZeRO-2/3: acc = s_0 + s_1 + ...  (s_m: rank-order sum of micro-batch m),
 *             then g = acc / D. */

/* ZeRO-1 local accumulation of micro-batch `micro` (0-based): for every rank
 * r and flat index i, acc_replicas[r][i] = x (micro 0) or acc + x (binary32),
 * x = grad_replicas[r][i] (padding reads 0).  acc_replicas: N_d fp32 buffers
 * of Psi_pad elements.  Stage 1 only (ZERO_ERR_STATE otherwise). */
zero_status_t zero_accumulate_grads(const zero_layout* L, int32_t micro, const void* const* grad_replicas,
                                    float* const* acc_replicas, zero_stream_t stream);

/* ZeRO-1 reduce-scatter of the fp32 accumulators of one bucket after the
 * last micro-batch: s = A_0 + A_1 + ... in rank order, grad_shards[r][j] =
 * s / (N_d * n_micro * loss_scale), plus norm partials and the non-finite
 * flag (as zero_reduce_scatter).  Stage 1 only. */
zero_status_t zero_reduce_scatter_accumulated(const zero_layout* L, int32_t bucket, const float* const* acc_replicas,
                                              float* const* grad_shards, int32_t n_micro, zero_step_state* st,
                                              void* workspace, zero_stream_t stream);

/* ZeRO-2/3 reduce-scatter of micro-batch `micro` of n_micro into the fp32
 * shard accumulators (which become the averaged gradient on the last one):
 * s = rank-order sum; micro 0: acc = s; middle: acc = acc + s; last:
 * acc = (acc + s) / (N_d * n_micro * loss_scale), with norm partials and the
 * non-finite flag.  n_micro = 1 is zero_reduce_scatter.  Every bucket (unit)
 * is reduced once per micro-batch.  Stages 2-3 (ZERO_ERR_STATE otherwise). */
zero_status_t zero_reduce_scatter_micro(const zero_layout* L, int32_t bucket_or_unit, int32_t micro,
                                        int32_t n_micro, const void* const* grad_replicas, float* const* acc_shards,
                                        zero_step_state* st, void* workspace, zero_stream_t stream);

/* Micro-batch `micro` (0-based) of an optimizer step over n_micro
 * micro-batches, whose 16-bit gradients are in args->grad_replicas, issued
 * by the step executor with the calls above ([RN] §4.1-§4.3):
 *   ZeRO-1: zero_accumulate_grads into acc_replicas (N_d fp32 buffers of
 *     Psi_pad); the last micro-batch then reduce-scatters the accumulators
 *     bucket by bucket (zero_reduce_scatter_accumulated);
 *   ZeRO-2: zero_reduce_scatter_micro for every bucket, every micro-batch;
 *   ZeRO-3: every unit gathered forward and backward and reduced
 *     (zero_reduce_scatter_micro) every micro-batch;
 * and after the last micro-batch's reductions zero_grad_norm(DECIDE) and the
 * update, as zero_step's split step.  Requires args->fused = 0 when
 * n_micro > 1; n_micro = 1 is zero_step.  Bucket launches rotate over streams
 * and ZeRO-3 units use transient2 as in zero_step.  acc_replicas: ZeRO-1 with
 * n_micro > 1 only (else ignored).  Errors: micro out of [0, n_micro),
 * fused with n_micro > 1, missing accumulators (ZERO_ERR_INVALID), and those
 * of zero_step. */
zero_status_t zero_micro_step(const zero_layout* L, const zero_step_args* args, int32_t micro, int32_t n_micro,
                              float* const* acc_replicas, zero_stream_t stream);

/* Largest Psi_pad that zero_fused_step_noalloc accepts (64 Mi elements). */
#define ZERO_NOALLOC_MAX_ELEMS 67108864

/* zero_fused_step over the whole buffer (every bucket; for ZeRO-3 every unit,
 * last unit first), followed by zero_grad_norm(..., ZERO_NORM_AFTER_FUSED),
 * for callers that cannot provide a device workspace.  The pages have no
 * counterpart: this is a convenience of this library.
 *
 * Who needs it: code that may not allocate device memory when it runs, for
 * example a plug-in inside a host application that owns all device memory
 * through its own pool, or a latency-critical loop where a cudaMalloc (which
 * can synchronise the device) is not allowed.  Instead of a caller workspace,
 * the norm scratch lives in a fixed array compiled into the library: 8 MiB +
 * 8 KiB of device memory that every GPU loading the library keeps until the
 * process exits.  The call itself allocates nothing.
 *
 * Limits and behaviour:
 *   - Psi_pad must not exceed ZERO_NOALLOC_MAX_ELEMS, else ZERO_ERR_INVALID
 *     (nothing is launched).  Stage 0: ZERO_ERR_STATE.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it with the id of the current context;
 *     make that first call before any stream capture begins.  A later call
 *     under another context of that device (after cudaDeviceReset) looks the
 *     address up again.
 *   - All calls share the array and it keeps the last call's contents;
 *     nothing needs clearing, because each call writes every slot before it
 *     reads it.  Calls that overlap on the GPU (other streams, other host
 *     threads) race on the array: serialise them.
 *   - Arguments, outputs and the update are those of zero_fused_step (no
 *     clipping, no loss-scale skip); ZeRO-3 requires ZERO_OUT_SHARDS. */
zero_status_t zero_fused_step_noalloc(const zero_layout* L, const zero_adamw_hp* hp,
                                      const void* const* grad_replicas, float* const* master,
                                      float* const* m, float* const* v, zero_step_state* st,
                                      void* const* param16_out, int32_t out_kind,
                                      zero_stream_t stream);

/* Cap on the CTAs of every later launch by this library (process-wide;
 * 0 = no cap: each kernel's own persistent grid, one full wave of CTAs or,
 * where that measured faster on GB300, fewer CTAs per SM).  For overlapping
 * the library's memory-bound kernels with other work on another stream
 * (ZeRO-3 prefetch under a layer's compute): a full-wave grid occupies every
 * SM, so concurrent kernels would serialise behind it.  Results do not depend
 * on the cap.  Returns the previous value. */
int32_t zero_set_max_ctas(int32_t max_ctas);

/* Message for the last failing call on this thread ("" if none). */
const char* zero_last_error(void);

/* Number of device kernels the library launched on this thread since the
 * last reset (for launch accounting in benchmarks). */
int64_t zero_launch_count(int32_t reset);

/* Bounds-checked builds.  A build compiled with -DZK_CHECKED (the build
 * script's checked=True, libzero_checked.so) tests every global access of
 * every kernel against the extent the layout gives its buffer (16-bit
 * replicas and accumulators: Psi_pad elements; fp32 shards and 16-bit
 * shards: S; a ZeRO-3 transient: the unit's real size; norm partials:
 * Psi_pad / 32; a rank index: N_d).  An access outside is skipped, never
 * made, and counted; nothing traps.  This stands in for a memory checker
 * ("the kernel reads and writes only inside the buffers the header
 * promises").  The normal build compiles the checks out.
 *   zero_checked_build: 1 for a checked build, 0 otherwise.
 *   zero_bounds_violations: *count = accesses skipped on the current device
 *     since the last reset (0 in a normal build); reset != 0 zeroes the count.
 *     Synchronises the device.  ZERO_ERR_CUDA if reading the count fails.
 *   zero_checked_set_slack: a test hook of checked builds: every extent the
 *     launches check against is `elems` elements short of the real one, so
 *     the last accesses of each buffer are reported and skipped while the
 *     buffers stay whole.  elems >= 0; returns ZERO_ERR_STATE in a normal
 *     build. */
int32_t zero_checked_build(void);
zero_status_t zero_bounds_violations(int64_t* count, int32_t reset);
zero_status_t zero_checked_set_slack(int64_t elems);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_H */
