// Host-side layout of the flat parameter buffer: flatten, pad, shard, bucket,
// ZeRO-3 units, and the per-rank memory / communication accounting.
//
// Flatten into one contiguous buffer: "ZeRO: Memory Optimizations Toward
// Training Trillion Parameter Models" reading notes, §2.2 and §5.2.  Equal
// 1/N_d split: "第 5 课：ZeRO 与 FSDP" §2 and the reading notes §4.1.  Fixed-size
// buckets reduced as backward fills them: mlqm.cn post "梯度桶化", reading notes
// §4.1-§4.2.  One unit per block plus a root unit: "別再複製本可分片的東西：ZeRO 與
// FSDP", FSDP section.  Memory M0..M3: "第 5 课" §2.  Volumes (N_d - 1)/N_d Psi
// per collective: "第 5 课" §3, reading notes §6.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "zero_internal.h"

namespace zero_detail {

static thread_local std::string g_last_error;
static thread_local int64_t g_launches = 0;

zero_status_t fail(zero_status_t code, const std::string& msg) {
    g_last_error = msg;
    return code;
}

void clear_error() { g_last_error.clear(); }

void count_launches(int64_t n) { g_launches += n; }

static std::atomic<int32_t> g_max_ctas{0};
int32_t max_ctas() { return g_max_ctas.load(std::memory_order_relaxed); }

int64_t partials_count(const zero_layout* L) { return L->psi_pad / kGroup; }

static int64_t round_up(int64_t x, int64_t m) { return ((x + m - 1) / m) * m; }

// Largest Psi and pad quantum accepted (the kernels' vector counters need
// Psi_pad / 8 < 2^31 in any case); it keeps every size sum inside int64.
static constexpr int64_t kMaxElems = (int64_t)1 << 34;

int64_t workspace_bytes(const zero_layout* L) {
    int64_t p = round_up(partials_count(L) * (int64_t)sizeof(float), 256);
    return p + round_up((int64_t)kNormBlocks * (int64_t)sizeof(double), 256);
}

}  // namespace zero_detail

using namespace zero_detail;

extern "C" const char* zero_last_error(void) { return g_last_error.c_str(); }

extern "C" int32_t zero_set_max_ctas(int32_t n) {
    return g_max_ctas.exchange(n < 0 ? 0 : n, std::memory_order_relaxed);
}

extern "C" int64_t zero_launch_count(int32_t reset) {
    int64_t n = g_launches;
    if (reset) g_launches = 0;
    return n;
}

// ---------------------------------------------------------------------------
// Bounds-checked builds (-DZK_CHECKED): the registry of per-translation-unit
// counters and the extent slack of the test hook.
// ---------------------------------------------------------------------------
namespace zero_detail {
static std::mutex& bounds_mu() {
    static std::mutex mu;
    return mu;
}
static std::vector<BoundsReader>& bounds_readers() {
    static std::vector<BoundsReader> v;
    return v;
}
void register_bounds_reader(BoundsReader fn) {
    std::lock_guard<std::mutex> lock(bounds_mu());
    bounds_readers().push_back(fn);
}
static std::atomic<int64_t> g_check_slack{0};
int64_t check_slack() { return g_check_slack.load(std::memory_order_relaxed); }
}  // namespace zero_detail

extern "C" int32_t zero_checked_build(void) {
#ifdef ZK_CHECKED
    return 1;
#else
    return 0;
#endif
}

extern "C" zero_status_t zero_bounds_violations(int64_t* count, int32_t reset) {
    clear_error();
    if (!count) return fail(ZERO_ERR_INVALID, "zero_bounds_violations: NULL output");
    *count = 0;
    std::lock_guard<std::mutex> lock(bounds_mu());
    for (BoundsReader fn : bounds_readers()) {
        const int e = fn(count, reset != 0);
        if (e != 0) return fail(ZERO_ERR_CUDA, "zero_bounds_violations: reading a device counter failed");
    }
    return ZERO_OK;
}

extern "C" zero_status_t zero_checked_set_slack(int64_t elems) {
    clear_error();
#ifdef ZK_CHECKED
    if (elems < 0) return fail(ZERO_ERR_INVALID, "zero_checked_set_slack: elems must be >= 0");
    g_check_slack.store(elems, std::memory_order_relaxed);
    return ZERO_OK;
#else
    (void)elems;
    return fail(ZERO_ERR_STATE, "zero_checked_set_slack: not a bounds-checked build");
#endif
}

extern "C" zero_status_t zero_layout_init(const int64_t* numels, int32_t n_tensors,
                                          const int32_t* unit_of_tensor, int32_t n_d,
                                          int32_t stage, int64_t pad_multiple,
                                          int64_t bucket_elems, zero_dtype_t dtype,
                                          zero_layout** out) {
    clear_error();
    if (!out || !numels || n_tensors <= 0) return fail(ZERO_ERR_INVALID, "layout: null argument or no tensors");
    if (n_d < 1 || n_d > ZERO_MAX_RANKS) return fail(ZERO_ERR_INVALID, "layout: n_d must be in 1..64");
    if (stage < 0 || stage > 3) return fail(ZERO_ERR_INVALID, "layout: stage must be 0..3");
    if (dtype != ZERO_BF16 && dtype != ZERO_FP16) return fail(ZERO_ERR_INVALID, "layout: dtype must be bf16 or fp16");
    const int64_t quantum = (int64_t)n_d * 128;
    int64_t q = pad_multiple > 0 ? pad_multiple : quantum;
    if (pad_multiple < 0 || q % quantum != 0 || q > kMaxElems)
        return fail(ZERO_ERR_INVALID, "layout: pad_multiple must be 0 or a positive multiple of n_d*128 (<= 2^34)");
    if (bucket_elems > 0 && bucket_elems % kGroup != 0)
        return fail(ZERO_ERR_INVALID, "layout: bucket_elems must be <= 0 or a multiple of 32");
    if (stage == 3 && !unit_of_tensor) return fail(ZERO_ERR_INVALID, "layout: stage 3 needs unit_of_tensor");

    zero_layout* L = new (std::nothrow) zero_layout();
    if (!L) return fail(ZERO_ERR_NOMEM, "layout: out of host memory");
    L->n_d = n_d;
    L->stage = stage;
    L->dtype = (int32_t)dtype;
    L->q = q;
    L->bucket_elems = bucket_elems;
    L->numels.assign(numels, numels + n_tensors);
    L->tensor_offset.assign(n_tensors, 0);
    int64_t psi = 0;
    for (int32_t t = 0; t < n_tensors; ++t) {
        if (numels[t] <= 0) {
            delete L;
            return fail(ZERO_ERR_INVALID, "layout: every tensor needs numel > 0");
        }
        if (numels[t] > kMaxElems - psi) {  // also keeps every later sum and rounding inside int64
            delete L;
            return fail(ZERO_ERR_INVALID, "layout: Psi too large (> 2^34 elements)");
        }
        psi += numels[t];
    }
    L->psi = psi;

    if (stage == 3) {
        int32_t n_units = 0;
        for (int32_t t = 0; t < n_tensors; ++t) {
            // no unit may be empty, so every id is below the tensor count
            if (unit_of_tensor[t] < 0 || unit_of_tensor[t] >= n_tensors) {
                delete L;
                return fail(ZERO_ERR_INVALID, "layout: unit ids must lie in 0..n_tensors-1");
            }
            n_units = std::max(n_units, unit_of_tensor[t] + 1);
        }
        std::vector<int64_t> real(n_units, 0);
        for (int32_t t = 0; t < n_tensors; ++t) real[unit_of_tensor[t]] += numels[t];
        for (int32_t u = 0; u < n_units; ++u) {
            if (real[u] == 0) {
                delete L;
                return fail(ZERO_ERR_INVALID, "layout: unit ids must cover 0..U-1 with no empty unit");
            }
        }
        std::vector<std::vector<int32_t>> members(n_units);  // tensors of each unit, in declaration order
        for (int32_t t = 0; t < n_tensors; ++t) members[unit_of_tensor[t]].push_back(t);
        int64_t off = 0, base = 0;
        for (int32_t u = 0; u < n_units; ++u) {
            int64_t r = 0;
            for (int32_t t : members[u]) {
                L->tensor_offset[t] = off + r;
                r += numels[t];
            }
            zero_segment s;
            s.offset = off;
            s.real = r;
            s.padded = round_up(r, q);
            s.shard = s.padded / n_d;
            s.shard_base = base;
            L->segs.push_back(s);
            L->buckets.emplace_back(s.offset, s.offset + s.padded);
            L->bucket_seg.push_back(u);
            off += s.padded;
            base += s.shard;
        }
        L->psi_pad = off;
        L->shard_len = base;
    } else {
        int64_t off = 0;
        for (int32_t t = 0; t < n_tensors; ++t) {
            L->tensor_offset[t] = off;
            off += numels[t];
        }
        zero_segment s;
        s.offset = 0;
        s.real = psi;
        s.padded = round_up(psi, q);
        s.shard = s.padded / n_d;
        s.shard_base = 0;
        L->segs.push_back(s);
        L->psi_pad = s.padded;
        L->shard_len = s.shard;
        if (bucket_elems <= 0 || bucket_elems >= L->psi_pad) {
            L->buckets.emplace_back(0, L->psi_pad);
            L->bucket_seg.push_back(0);
        } else {
            for (int64_t b = 0; b < L->psi_pad; b += bucket_elems) {
                L->buckets.emplace_back(b, std::min(b + bucket_elems, L->psi_pad));
                L->bucket_seg.push_back(0);
            }
        }
    }
    // Kernels index 8-element vectors with 32-bit grid-stride counters; keep
    // the vector count below 2^31 so a counter never wraps.
    if (L->psi_pad / 8 >= (int64_t)1 << 31) {
        delete L;
        return fail(ZERO_ERR_INVALID, "layout: Psi_pad too large (>= 2^34 elements)");
    }
    *out = L;
    return ZERO_OK;
}

extern "C" zero_status_t zero_layout_query(const zero_layout* L, zero_layout_info* o) {
    clear_error();
    if (!L || !o) return fail(ZERO_ERR_INVALID, "query: null argument");
    std::memset(o, 0, sizeof(*o));
    o->n_d = L->n_d;
    o->stage = L->stage;
    o->dtype = L->dtype;
    o->n_tensors = (int32_t)L->numels.size();
    o->n_buckets = (int32_t)L->buckets.size();
    o->n_units = (int32_t)L->segs.size();
    o->psi = L->psi;
    o->psi_pad = L->psi_pad;
    o->q = L->q;
    o->bucket_elems = L->bucket_elems;
    o->shard_len = L->shard_len;
    int64_t maxu = 0;
    for (const auto& s : L->segs) maxu = std::max(maxu, s.padded);
    o->max_unit_padded = maxu;
    const int64_t S = L->shard_len, P = L->psi_pad;
    switch (L->stage) {
        case 0: o->mem_formula = 16 * P; break;
        case 1: o->mem_formula = 4 * P + 12 * S; break;
        case 2: o->mem_formula = 2 * P + 14 * S; break;
        default: o->mem_formula = 16 * S; break;
    }
    o->mem_state = 12 * S;
    o->mem_gshard = 4 * S;
    o->mem_transient = L->stage == 3 ? 2 * maxu : 0;
    o->mem_peak = o->mem_formula + o->mem_transient;
    const int64_t one = (int64_t)(L->n_d - 1) * S;
    if (L->stage == 0) {
        o->comm_allreduce = 2 * one;
        o->comm_total = 2 * one;
    } else if (L->stage == 3) {
        o->comm_rs = one;
        o->comm_ag_fwd = one;
        o->comm_ag_bwd = one;
        o->comm_total = 3 * one;
    } else {
        o->comm_rs = one;
        o->comm_ag = one;
        o->comm_total = 2 * one;
    }
    o->workspace_bytes = workspace_bytes(L);
    return ZERO_OK;
}

extern "C" zero_status_t zero_layout_bucket(const zero_layout* L, int32_t b, int64_t* begin,
                                            int64_t* end) {
    clear_error();
    if (!L || !begin || !end) return fail(ZERO_ERR_INVALID, "bucket: null argument");
    if (b < 0 || b >= (int32_t)L->buckets.size()) return fail(ZERO_ERR_INVALID, "bucket: index out of range");
    *begin = L->buckets[b].first;
    *end = L->buckets[b].second;
    return ZERO_OK;
}

extern "C" zero_status_t zero_layout_unit(const zero_layout* L, int32_t u, zero_unit_info* o) {
    clear_error();
    if (!L || !o) return fail(ZERO_ERR_INVALID, "unit: null argument");
    if (u < 0 || u >= (int32_t)L->segs.size()) return fail(ZERO_ERR_INVALID, "unit: index out of range");
    const zero_segment& s = L->segs[u];
    o->offset = s.offset;
    o->real = s.real;
    o->padded = s.padded;
    o->shard = s.shard;
    o->shard_base = s.shard_base;
    return ZERO_OK;
}

extern "C" zero_status_t zero_layout_tensor_offset(const zero_layout* L, int32_t t, int64_t* offset) {
    clear_error();
    if (!L || !offset) return fail(ZERO_ERR_INVALID, "tensor: null argument");
    if (t < 0 || t >= (int32_t)L->numels.size()) return fail(ZERO_ERR_INVALID, "tensor: index out of range");
    *offset = L->tensor_offset[t];
    return ZERO_OK;
}

extern "C" void zero_layout_destroy(zero_layout* L) { delete L; }

// Where flat index i lives: (rank, shard offset, elements left in that shard).
static void locate(const zero_layout* L, int64_t i, int32_t* rank, int64_t* off, int64_t* left) {
    size_t lo = 0, hi = L->segs.size();
    while (hi - lo > 1) {  // last segment with offset <= i
        size_t mid = (lo + hi) / 2;
        if (L->segs[mid].offset <= i) lo = mid; else hi = mid;
    }
    const zero_segment& s = L->segs[lo];
    const int64_t k = i - s.offset;
    const int64_t r = k / s.shard;
    *rank = (int32_t)r;
    *off = s.shard_base + (k - r * s.shard);
    *left = s.shard - (k - r * s.shard);
}

extern "C" zero_status_t zero_reshard_plan(const zero_layout* src, const zero_layout* dst,
                                           zero_copy_segment* out, int64_t capacity, int64_t* count) {
    clear_error();
    if (!src || !dst || !count) return fail(ZERO_ERR_INVALID, "reshard: null argument");
    if (src->stage == 0 || dst->stage == 0) return fail(ZERO_ERR_INVALID, "reshard: stage 0 has no shards");
    if (src->numels != dst->numels) return fail(ZERO_ERR_INVALID, "reshard: layouts hold different tensors");
    int64_t n = 0;
    bool have = false;
    zero_copy_segment cur{};
    auto emit = [&](const zero_copy_segment& g) {
        if (have && cur.src_rank == g.src_rank && cur.dst_rank == g.dst_rank &&
            cur.src_off + cur.len == g.src_off && cur.dst_off + cur.len == g.dst_off) {
            cur.len += g.len;
            return;
        }
        if (have) {
            if (out && n < capacity) out[n] = cur;
            ++n;
        }
        cur = g;
        have = true;
    };
    for (size_t t = 0; t < src->numels.size(); ++t) {
        const int64_t total = src->numels[t];
        int64_t pos = 0;
        while (pos < total) {
            zero_copy_segment g{};
            int64_t ls, ld;
            locate(src, src->tensor_offset[t] + pos, &g.src_rank, &g.src_off, &ls);
            locate(dst, dst->tensor_offset[t] + pos, &g.dst_rank, &g.dst_off, &ld);
            g.len = std::min(std::min(ls, ld), total - pos);
            emit(g);
            pos += g.len;
        }
    }
    if (have) {
        if (out && n < capacity) out[n] = cur;
        ++n;
    }
    *count = n;
    if (out && n > capacity) return fail(ZERO_ERR_INVALID, "reshard: capacity too small");
    return ZERO_OK;
}
