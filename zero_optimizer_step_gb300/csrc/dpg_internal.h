// dpg_internal.h -- private declarations shared by the planner (host C++) and
// the CUDA translation unit of libdpg.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <mutex>
#include <string>
#include <vector>

#include "dpg.h"
#include <nvtx3/nvToolsExt.h>

namespace dpg {

// NVTX range around one C-ABI call, so that a timeline (Nsight Systems, or
// any NVTX-aware tool) shows each call by name; a no-op with no tool attached.
struct Trace {
    explicit Trace(const char* name) { nvtxRangePushA(name); }
    ~Trace() { nvtxRangePop(); }
    Trace(const Trace&) = delete;
    Trace& operator=(const Trace&) = delete;
};

// Geometry of the fused pass.  One thread owns one 8-element vector (16 bytes
// of bf16 gradient per replica, 32 bytes of each fp32 state array); a CTA of
// kThreads threads covers one tile of kTile elements.  Tiles never straddle a
// bucket (the last tile of a bucket may be partial), so every tile's norm
// partials belong to exactly one bucket.  One 512-thread CTA per SM (the
// R = 8 kernel needs ~92 registers per thread) measured 0.3 % faster than
// two 256-thread CTAs and 1-3 % faster than higher occupancy at fewer
// registers, on the 1B workload.
constexpr int kVec = 8;
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int64_t kTile = int64_t(kThreads) * kVec;

// Pack/unpack work is cut into items of at most kPackChunk elements; one CTA
// copies one item.  kPackPtrs parameter pointers travel in one launch's
// argument block.
constexpr int64_t kPackChunk = 65536;
constexpr int kPackPtrs = 1024;

// The per-bucket norm of a chunked launch is summed by one finalize CTA per
// segment of at most kSegTiles tiles of one bucket (8192 chunk partials: one
// round of 8 loads for each of its 1024 threads); the last CTA of a bucket
// adds its segments' sums.
constexpr int64_t kSegTiles = 2048;
// A bucket of at most kShortTiles tiles (<= 1024 chunk partials) is summed by
// one warp instead of a CTA: many small buckets then cost a few warps each.
constexpr int64_t kShortTiles = 256;

struct PackItem {
    int32_t param;     // registration index of the parameter
    int32_t reserved;
    int64_t src_off;   // element offset inside the parameter
    int64_t flat_off;  // element offset in the flat buffer
    int64_t count;     // elements copied
    int64_t tail;      // zero elements written right after the copy (pack, import)
    int64_t canon_off; // element offset in the canonical (registration-order) layout
};

struct Plan {
    int32_t n_params = 0, n_buckets = 0, R = 1;
    int64_t cap_bytes = 0, total_padded = 0, n_tiles = 0;
    std::vector<int64_t> numels, param_offset;
    int64_t canon_total = 0;             // sum of numels
    std::vector<int32_t> param_bucket;
    std::vector<int64_t> bucket_offset;  // n_buckets + 1 entries, last = total_padded
    std::vector<int64_t> tile_begin;     // n_buckets + 1 entries, last = n_tiles
    std::vector<PackItem> items;         // flat (= descending registration) order

    // device copy, made on first device use
    std::mutex mu;
    int device = -1;
    int64_t* d_bucket_offset = nullptr;
    int64_t* d_tile_begin = nullptr;
    PackItem* d_items = nullptr;
    // norm scratch: per-(CTA, bucket visit) partials of one fused launch
    void* d_vis = nullptr;          // one allocation, sections below
    double* d_vis_sq = nullptr;     // cap_visits * kWarps
    int32_t* d_vis_nf = nullptr;    // cap_visits * kWarps
    int32_t* d_vis_bucket = nullptr;// cap_visits
    int32_t* d_vis_count = nullptr; // cap_ctas
    int64_t cap_visits = 0;
    int32_t cap_ctas = 0;
    // chunked launches: tile spans (n_tiles) and per-chunk norm partials
    // (chunks_per_tile * n_tiles each), one allocation
    void* d_chunk = nullptr;
    int64_t* d_tile_span = nullptr;     // 2 per tile: first element, end of its bucket
    double* d_chunk_sq = nullptr;
    int32_t* d_chunk_nf = nullptr;
    // chunk-norm finalize: segments of <= kSegTiles tiles, bucket b owning
    // segments [seg_first[b], seg_first[b + 1]); per-segment sums; per-bucket
    // arrival counters (zero between launches: the last CTA resets its own)
    std::vector<int32_t> seg_first;   // n_buckets + 1 (host copy)
    int32_t n_seg = 0;
    void* d_seg = nullptr;            // one allocation, sections below
    int32_t* d_seg_first = nullptr;   // n_buckets + 1
    int32_t* d_seg_bucket = nullptr;  // n_seg
    double* d_seg_sq = nullptr;       // n_seg
    long long* d_seg_nf = nullptr;    // n_seg
    int32_t* d_bucket_done = nullptr; // n_buckets
    // short buckets (<= kShortTiles tiles) are finalized by one warp each,
    // the segments of the other buckets by one CTA each; both lists ascend,
    // and the host prefixes give each bucket range's slice of them
    std::vector<int32_t> short_first; // n_buckets + 1: short buckets before b
    std::vector<int32_t> long_first;  // n_buckets + 1: long-bucket segments before b
    int32_t* d_short_bucket = nullptr;// short bucket ids
    int32_t* d_long_seg = nullptr;    // segment ids of the long buckets
    // global-norm clipping: per-bucket fp64 squared norms and the coefficient
    void* d_clip = nullptr;
    double* d_bucket_sq64 = nullptr;  // n_buckets + 1
    float* d_clip_coef = nullptr;     // 1
    int32_t* d_status = nullptr;      // status word of the staged pass (0 = OK)
    unsigned long long* d_debug = nullptr;  // first failed index check (checking builds)
};

// thread-local error message
int fail(int status, const char* fmt, ...);
void clear_error();

// device side (dpg_runtime.cu)
int upload(Plan& p);
void release_device(Plan& p);

}  // namespace dpg

struct dpg_plan {
    dpg::Plan p;
};
