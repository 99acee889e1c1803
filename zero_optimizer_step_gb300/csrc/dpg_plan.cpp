// dpg_plan.cpp -- host bucket planner and plan queries of libdpg.
//
// Gradient bucketing ("Parallelisms" -- Data parallel, Gradient bucketing;
// "Distributed Training and Parallelism" -- Data parallelism and the global
// gradient): buckets of later layers become ready first in backward, so the
// parameters are walked in reverse registration order and packed greedily
// into flat buffers capped at cap_bytes of bf16 gradient.  Each gradient is a
// view into a slice of its bucket ("Parallelisms" -- FSDP / Flat parameter);
// each bucket splits into R equal shards, shard r owned by rank r
// ("Parallelisms" -- ZeRO-2).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <new>

#include "dpg_internal.h"

namespace dpg {

static thread_local std::string t_error;

int fail(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_error = buf;
    return status;
}

void clear_error() { t_error.clear(); }

static int64_t round_up(int64_t x, int64_t unit) { return (x + unit - 1) / unit * unit; }

// Fill p.param_bucket / p.param_offset / p.bucket_offset from p.numels.
static void place(Plan& p) {
    const int64_t vec = 8;
    const int64_t shard_unit = vec * p.R;
    int64_t base = 0;      // flat offset of the open bucket
    int64_t fill = 0;      // end of the last slice in the open bucket (elements)
    int32_t open_members = 0;
    p.bucket_offset.clear();
    for (int32_t q = p.n_params - 1; q >= 0; --q) {
        const int64_t n = p.numels[q];
        int64_t at = round_up(fill, vec);
        const bool holds_elements = fill > 0;
        if (holds_elements && n > 0 && (at + n) * 2 > p.cap_bytes) {
            p.bucket_offset.push_back(base);
            base += round_up(fill, shard_unit);
            fill = 0;
            open_members = 0;
            at = 0;
        }
        p.param_bucket[q] = int32_t(p.bucket_offset.size());
        p.param_offset[q] = base + at;
        fill = at + n;
        ++open_members;
    }
    if (open_members > 0) {
        p.bucket_offset.push_back(base);
        base += round_up(fill, shard_unit);
    }
    p.n_buckets = int32_t(p.bucket_offset.size());
    p.total_padded = base;
    p.bucket_offset.push_back(base);  // sentinel: end of the last bucket
}

// Tiles of the fused pass: ceil(padded_b / kTile) per bucket.
static void tile(Plan& p) {
    p.tile_begin.assign(size_t(p.n_buckets) + 1, 0);
    for (int32_t b = 0; b < p.n_buckets; ++b) {
        const int64_t padded = p.bucket_offset[b + 1] - p.bucket_offset[b];
        p.tile_begin[b + 1] = p.tile_begin[b] + (padded + kTile - 1) / kTile;
    }
    p.n_tiles = p.tile_begin[p.n_buckets];
}

// Pack items in flat order; the last item of every parameter zero-fills the
// gap up to the next slice (or to the end of its bucket).
static void itemise(Plan& p) {
    p.items.clear();
    std::vector<int64_t> canon(size_t(p.n_params) + 1, 0);
    for (int32_t q = 0; q < p.n_params; ++q) canon[q + 1] = canon[q] + p.numels[q];
    p.canon_total = canon[p.n_params];
    for (int32_t q = p.n_params - 1; q >= 0; --q) {
        const int64_t start = p.param_offset[q];
        const int64_t n = p.numels[q];
        int64_t next;
        if (q > 0 && p.param_bucket[q - 1] == p.param_bucket[q]) {
            next = p.param_offset[q - 1];
        } else {
            next = p.bucket_offset[p.param_bucket[q] + 1];
        }
        int64_t off = 0;
        do {
            PackItem it{};
            it.param = q;
            it.src_off = off;
            it.flat_off = start + off;
            it.count = std::min<int64_t>(kPackChunk, n - off);
            off += it.count;
            it.tail = (off == n) ? next - (start + n) : 0;
            it.canon_off = canon[q] + it.src_off;
            p.items.push_back(it);
        } while (off < n);
    }
}

}  // namespace dpg

using dpg::fail;

extern "C" {

int dpg_abi_version(void) { return DPG_ABI_VERSION; }

const char* dpg_last_error(void) { return dpg::t_error.c_str(); }

const char* dpg_status_string(int status) {
    switch (status) {
        case DPG_OK: return "DPG_OK";
        case DPG_ERR_INVALID_ARG: return "DPG_ERR_INVALID_ARG";
        case DPG_ERR_ZERO_TOKENS: return "DPG_ERR_ZERO_TOKENS";
        case DPG_ERR_MISALIGNED: return "DPG_ERR_MISALIGNED";
        case DPG_ERR_CUDA: return "DPG_ERR_CUDA";
        case DPG_ERR_DEVICE_TIMEOUT: return "DPG_ERR_DEVICE_TIMEOUT";
        case DPG_ERR_OOM: return "DPG_ERR_OOM";
        default: return "DPG_ERR_UNKNOWN";
    }
}

int dpg_plan_buckets(const int64_t* numels, int32_t n_params, int64_t cap_bytes, int32_t R,
                     dpg_plan_t** out) {
    dpg::clear_error();
    if (!out) return fail(DPG_ERR_INVALID_ARG, "dpg_plan_buckets: out is NULL");
    *out = nullptr;
    if (n_params < 0) return fail(DPG_ERR_INVALID_ARG, "dpg_plan_buckets: n_params < 0");
    if (n_params > 0 && !numels) return fail(DPG_ERR_INVALID_ARG, "dpg_plan_buckets: numels is NULL");
    if (cap_bytes <= 0) return fail(DPG_ERR_INVALID_ARG, "dpg_plan_buckets: cap_bytes must be > 0");
    if (R < 1 || R > DPG_MAX_REPLICAS)
        return fail(DPG_ERR_INVALID_ARG, "dpg_plan_buckets: R=%d outside [1, %d]", R,
                    DPG_MAX_REPLICAS);
    int64_t sum = 0;
    for (int32_t q = 0; q < n_params; ++q) {
        if (numels[q] < 0)
            return fail(DPG_ERR_INVALID_ARG, "dpg_plan_buckets: numels[%d] < 0", q);
        // each slice adds at most 7 alignment elements and each bucket at most
        // 8R-1 padding elements; keep the flat size far from int64 overflow
        if (numels[q] > (int64_t(1) << 56) || (sum += numels[q] + 8 + 8 * R) > (int64_t(1) << 58))
            return fail(DPG_ERR_INVALID_ARG, "dpg_plan_buckets: total size too large");
    }
    dpg_plan* h = new (std::nothrow) dpg_plan();
    if (!h) return fail(DPG_ERR_OOM, "dpg_plan_buckets: out of host memory");
    try {
        dpg::Plan& p = h->p;
        p.n_params = n_params;
        p.R = R;
        p.cap_bytes = cap_bytes;
        p.numels.assign(numels, numels + n_params);
        p.param_bucket.assign(size_t(n_params), 0);
        p.param_offset.assign(size_t(n_params), 0);
        dpg::place(p);
        dpg::tile(p);
        dpg::itemise(p);
    } catch (const std::bad_alloc&) {
        delete h;
        return fail(DPG_ERR_OOM, "dpg_plan_buckets: out of host memory");
    }
    *out = h;
    return DPG_OK;
}

int dpg_plan_shards(const dpg_plan_t* plan, dpg_plan_t** out) {
    dpg::clear_error();
    if (!out) return fail(DPG_ERR_INVALID_ARG, "dpg_plan_shards: out is NULL");
    *out = nullptr;
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_plan_shards: plan is NULL");
    const dpg::Plan& g = plan->p;
    // one "parameter" per bucket of the global plan, registered in reverse
    // bucket order so that the planner (which walks registration order
    // backwards) places shard 0 first; a 2-byte cap keeps each alone
    std::vector<int64_t> numels;
    try {
        numels.assign(size_t(g.n_buckets), 0);
    } catch (const std::bad_alloc&) {
        return fail(DPG_ERR_OOM, "dpg_plan_shards: out of host memory");
    }
    for (int32_t b = 0; b < g.n_buckets; ++b)
        numels[size_t(g.n_buckets - 1 - b)] = (g.bucket_offset[b + 1] - g.bucket_offset[b]) / g.R;
    dpg_plan_t* h = nullptr;
    const int st = dpg_plan_buckets(numels.data(), g.n_buckets, 2, g.R, &h);
    if (st != DPG_OK) return st;
    if (h->p.n_buckets != g.n_buckets) {
        dpg_plan_destroy(h);
        return fail(DPG_ERR_INVALID_ARG, "dpg_plan_shards: a bucket of the plan holds no element");
    }
    *out = h;
    return DPG_OK;
}

void dpg_plan_destroy(dpg_plan_t* plan) {
    if (!plan) return;
    dpg::release_device(plan->p);
    delete plan;
}

int dpg_plan_info(const dpg_plan_t* plan, int32_t* n_params, int32_t* n_buckets,
                  int64_t* total_padded, int32_t* R) {
    dpg::clear_error();
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_plan_info: plan is NULL");
    if (n_params) *n_params = plan->p.n_params;
    if (n_buckets) *n_buckets = plan->p.n_buckets;
    if (total_padded) *total_padded = plan->p.total_padded;
    if (R) *R = plan->p.R;
    return DPG_OK;
}

int dpg_plan_bucket(const dpg_plan_t* plan, int32_t b, int64_t* offset, int64_t* padded_numel,
                    int64_t* shard_numel) {
    dpg::clear_error();
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_plan_bucket: plan is NULL");
    const dpg::Plan& p = plan->p;
    if (b < 0 || b >= p.n_buckets)
        return fail(DPG_ERR_INVALID_ARG, "dpg_plan_bucket: bucket %d outside [0, %d)", b,
                    p.n_buckets);
    const int64_t padded = p.bucket_offset[b + 1] - p.bucket_offset[b];
    if (offset) *offset = p.bucket_offset[b];
    if (padded_numel) *padded_numel = padded;
    if (shard_numel) *shard_numel = padded / p.R;
    return DPG_OK;
}

int dpg_plan_param(const dpg_plan_t* plan, int32_t q, int32_t* bucket, int64_t* offset,
                   int64_t* numel) {
    dpg::clear_error();
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_plan_param: plan is NULL");
    const dpg::Plan& p = plan->p;
    if (q < 0 || q >= p.n_params)
        return fail(DPG_ERR_INVALID_ARG, "dpg_plan_param: parameter %d outside [0, %d)", q,
                    p.n_params);
    if (bucket) *bucket = p.param_bucket[q];
    if (offset) *offset = p.param_offset[q];
    if (numel) *numel = p.numels[q];
    return DPG_OK;
}

int dpg_plan_export(const dpg_plan_t* plan, int32_t* param_bucket, int64_t* param_offset,
                    int64_t* bucket_offset, int64_t* bucket_padded) {
    dpg::clear_error();
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_plan_export: plan is NULL");
    const dpg::Plan& p = plan->p;
    if (param_bucket) std::copy(p.param_bucket.begin(), p.param_bucket.end(), param_bucket);
    if (param_offset) std::copy(p.param_offset.begin(), p.param_offset.end(), param_offset);
    for (int32_t b = 0; b < p.n_buckets; ++b) {
        if (bucket_offset) bucket_offset[b] = p.bucket_offset[b];
        if (bucket_padded) bucket_padded[b] = p.bucket_offset[b + 1] - p.bucket_offset[b];
    }
    return DPG_OK;
}

}  // extern "C"
