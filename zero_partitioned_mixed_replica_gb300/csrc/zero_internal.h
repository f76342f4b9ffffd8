// Internal declarations shared by libzero's translation units (host side).
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "zero.h"

struct zero_segment {
    int64_t offset;      // flat offset
    int64_t real;        // real elements
    int64_t padded;      // padded elements (multiple of q)
    int64_t shard;       // S_u = padded / n_d
    int64_t shard_base;  // offset inside every rank's shard
};

struct zero_layout {
    int32_t n_d = 0;
    int32_t stage = 0;
    int32_t dtype = 0;
    int64_t q = 0;
    int64_t bucket_elems = 0;
    int64_t psi = 0;
    int64_t psi_pad = 0;
    int64_t shard_len = 0;
    std::vector<int64_t> numels;
    std::vector<int64_t> tensor_offset;
    std::vector<zero_segment> segs;                     // 1 for stages 0-2, U for stage 3
    std::vector<std::pair<int64_t, int64_t>> buckets;   // stage 3: one per unit
    std::vector<int32_t> bucket_seg;                    // segment of each bucket
};

namespace zero_detail {
// Norm partials: one float per 32 flat elements, then NORM_BLOCKS doubles.
constexpr int64_t kGroup = 32;
constexpr int32_t kNormBlocks = 1024;
int64_t partials_count(const zero_layout* L);
int64_t workspace_bytes(const zero_layout* L);
zero_status_t fail(zero_status_t code, const std::string& msg);
void clear_error();
void count_launches(int64_t n);
int32_t max_ctas();
// Bounds-checked builds: each CUDA translation unit registers a reader of its
// device counter of skipped accesses (adds it to *out; reset zeroes it), and
// the launches shorten every extent by check_slack() elements (a test hook).
using BoundsReader = int (*)(int64_t* out, bool reset);
void register_bounds_reader(BoundsReader fn);
int64_t check_slack();
}  // namespace zero_detail
