// dpg_runtime.cu -- host runtime of libdpg: the plan's device tables and
// scratch, launch geometry, launch counting, the per-thread launch knobs, and
// the Adam constants and token normalisation every step computes on the host.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "dpg_host.h"

namespace dpg {

std::atomic<int64_t> g_launches{0};
thread_local cudaEvent_t t_fused_start = nullptr, t_fused_stop = nullptr;
thread_local int64_t t_staged_skip = -1;
thread_local int64_t t_staged_timeout_ns = 0;
thread_local int32_t t_fused_max_ctas = 0;
thread_local int32_t t_programmatic = 1;
thread_local int64_t t_debug_limit = -1;

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------
int sm_count(int dev, int* out) {
    static std::mutex mu;
    static std::map<int, int> cache;
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(dev);
    if (it == cache.end()) {
        int n = 0;
        DPG_CUDA_TRY(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev));
        it = cache.emplace(dev, n).first;
    }
    *out = it->second;
    return DPG_OK;
}

// One CTA per `work_ctas` unit of work: the streaming kernels (accumulate,
// all-gather, gathers, pack, state copy) keep more bytes in flight with many
// short CTAs, several resident per SM at different points of their loads and
// stores, than with a resident-sized grid that strides over the work.
int grid_cover(int64_t work_ctas, int* grid, const char* who) {
    if (work_ctas > 0x7FFFFFFF)
        return fail(DPG_ERR_INVALID_ARG, "%s: %lld CTAs in one launch", who, (long long)work_ctas);
    *grid = int(work_ctas > 0 ? work_ctas : 1);
    return DPG_OK;
}

// persistent-grid size: SM count x resident CTAs of `fn` (cached per device)
int grid_for(const void* fn, int threads, int dev, int64_t work_ctas, int* grid) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> cache;
    int sms = 0;
    int st = sm_count(dev, &sms);
    if (st != DPG_OK) return st;
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> g(mu);
        auto key = std::make_pair(fn, dev);
        auto it = cache.find(key);
        if (it == cache.end()) {
            DPG_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, 0));
            if (per_sm < 1) per_sm = 1;
            it = cache.emplace(key, per_sm).first;
        }
        per_sm = it->second;
    }
    const int64_t full = int64_t(sms) * per_sm;
    *grid = int(work_ctas < full ? (work_ctas > 0 ? work_ctas : 1) : full);
    return DPG_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int after_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(DPG_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return DPG_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }


VisLayout vis_layout(int64_t visits, int64_t ctas) {
    VisLayout L;
    L.sq = 0;
    L.nf = L.sq + round256(size_t(visits) * kWarps * sizeof(double));
    L.bucket = L.nf + round256(size_t(visits) * kWarps * sizeof(int32_t));
    L.count = L.bucket + round256(size_t(visits) * sizeof(int32_t));
    L.total = L.count + round256(size_t(ctas) * sizeof(int32_t));
    return L;
}

int upload(Plan& p) {
    std::lock_guard<std::mutex> g(p.mu);
    int dev = 0;
    DPG_CUDA_TRY(cudaGetDevice(&dev));
    if (p.device >= 0) {
        if (p.device != dev)
            return fail(DPG_ERR_INVALID_ARG,
                        "plan tables live on device %d but device %d is current", p.device, dev);
        return DPG_OK;
    }
    int sms = 0;
    int st = sm_count(dev, &sms);
    if (st != DPG_OK) return st;
    // A fused launch over tiles T of buckets B with G CTAs uses G * min(B,
    // ceil(T / G)) visit slots: at most T + G and at most G * B, G being at
    // most the resident CTAs of the device (2048 threads per SM).
    const int64_t cap_ctas = int64_t(sms) * (2048 / kThreads);
    // (the staged pass works on up to two units per tile: twice as many)
    int64_t cap_visits = 2 * p.n_tiles + cap_ctas;
    if (cap_ctas * p.n_buckets < cap_visits) cap_visits = cap_ctas * p.n_buckets;
    if (cap_visits < 1) cap_visits = 1;
    const VisLayout L = vis_layout(cap_visits, cap_ctas);

    const size_t nb1 = size_t(p.n_buckets) + 1;
    const size_t n_items = p.items.size() ? p.items.size() : 1;
    void *bo = nullptr, *tb = nullptr, *it = nullptr, *vis = nullptr;
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = cudaMalloc(&bo, nb1 * sizeof(int64_t));
    if (e == cudaSuccess) e = cudaMalloc(&tb, nb1 * sizeof(int64_t));
    if (e == cudaSuccess) e = cudaMalloc(&it, n_items * sizeof(PackItem));
    if (e == cudaSuccess) e = cudaMalloc(&vis, L.total);
    const size_t clip_sq_bytes = round256(nb1 * sizeof(double));
    void* clip = nullptr;
    if (e == cudaSuccess) e = cudaMalloc(&clip, clip_sq_bytes + 256);
    // chunked launches: tile spans, then the per-chunk norm partials
    const size_t n_tiles1 = size_t(p.n_tiles > 0 ? p.n_tiles : 1);
    const size_t n_chunks1 = n_tiles1 * kChunksPerTile;
    const size_t tb_bytes = round256(n_tiles1 * 2 * sizeof(int64_t));
    const size_t csq_bytes = round256(n_chunks1 * sizeof(double));
    void* chunk = nullptr;
    if (e == cudaSuccess) e = cudaMalloc(&chunk, tb_bytes + csq_bytes + n_chunks1 * sizeof(int32_t));
    // finalize segments: ceil(tiles / kSegTiles) per bucket, at least one;
    // short buckets (one segment of <= kShortTiles tiles) go to the warp list
    std::vector<int32_t> seg_first(nb1, 0), seg_bucket;
    std::vector<int32_t> short_first(nb1, 0), long_first(nb1, 0), short_bucket, long_seg;
    for (int32_t b = 0; b < p.n_buckets; ++b) {
        const int64_t nt = p.tile_begin[b + 1] - p.tile_begin[b];
        const int64_t ns = nt > 0 ? (nt + kSegTiles - 1) / kSegTiles : 1;
        const bool is_short = nt <= kShortTiles;
        if (is_short) short_bucket.push_back(b);
        for (int64_t k = 0; k < ns; ++k) {
            if (!is_short) long_seg.push_back(int32_t(seg_bucket.size()));
            seg_bucket.push_back(b);
        }
        seg_first[size_t(b) + 1] = int32_t(seg_bucket.size());
        short_first[size_t(b) + 1] = int32_t(short_bucket.size());
        long_first[size_t(b) + 1] = int32_t(long_seg.size());
    }
    const size_t n_seg1 = seg_bucket.empty() ? 1 : seg_bucket.size();
    const size_t sf_bytes = round256(nb1 * sizeof(int32_t));
    const size_t sb_bytes = round256(n_seg1 * sizeof(int32_t));
    const size_t ss_bytes = round256(n_seg1 * sizeof(double));
    const size_t sn_bytes = round256(n_seg1 * sizeof(long long));
    const size_t done_bytes = round256(nb1 * sizeof(int32_t));
    const size_t shb_bytes = round256(nb1 * sizeof(int32_t));     // short bucket ids
    const size_t lsg_bytes = round256(n_seg1 * sizeof(int32_t));  // long-bucket segment ids
    void* seg = nullptr;
    if (e == cudaSuccess)
        e = cudaMalloc(&seg, sf_bytes + sb_bytes + ss_bytes + sn_bytes + done_bytes + shb_bytes +
                                 lsg_bytes);
    unsigned char* sbase = static_cast<unsigned char*>(seg);
    unsigned char* shb = sbase + sf_bytes + sb_bytes + ss_bytes + sn_bytes + done_bytes;
    if (e == cudaSuccess)
        e = cudaMemcpy(sbase, seg_first.data(), nb1 * sizeof(int32_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !seg_bucket.empty())
        e = cudaMemcpy(sbase + sf_bytes, seg_bucket.data(), seg_bucket.size() * sizeof(int32_t),
                       cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
        e = cudaMemset(sbase + sf_bytes + sb_bytes + ss_bytes + sn_bytes, 0, done_bytes);
    if (e == cudaSuccess && !short_bucket.empty())
        e = cudaMemcpy(shb, short_bucket.data(), short_bucket.size() * sizeof(int32_t),
                       cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !long_seg.empty())
        e = cudaMemcpy(shb + shb_bytes, long_seg.data(), long_seg.size() * sizeof(int32_t),
                       cudaMemcpyHostToDevice);
    std::vector<int64_t> tile_span(2 * n_tiles1, 0);
    for (int32_t b = 0; b < p.n_buckets; ++b)
        for (int64_t t = p.tile_begin[b]; t < p.tile_begin[b + 1]; ++t) {
            tile_span[2 * size_t(t)] = p.bucket_offset[b] + (t - p.tile_begin[b]) * kTile;
            tile_span[2 * size_t(t) + 1] = p.bucket_offset[b + 1];
        }
    if (e == cudaSuccess)
        e = cudaMemcpy(chunk, tile_span.data(), tile_span.size() * sizeof(int64_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(bo, p.bucket_offset.data(), nb1 * sizeof(int64_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(tb, p.tile_begin.data(), nb1 * sizeof(int64_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !p.items.empty())
        e = cudaMemcpy(it, p.items.data(), p.items.size() * sizeof(PackItem), cudaMemcpyHostToDevice);
#ifdef DPG_DEBUG
    if (e == cudaSuccess) e = cudaMemset(static_cast<unsigned char*>(clip) + clip_sq_bytes + 192, 0, 8);
#endif
    if (e != cudaSuccess) {
        cudaFree(bo); cudaFree(tb); cudaFree(it); cudaFree(vis); cudaFree(clip); cudaFree(chunk);
        cudaFree(seg);
        cudaGetLastError();
        return fail(e == cudaErrorMemoryAllocation ? DPG_ERR_OOM : DPG_ERR_CUDA,
                    "plan upload: %s", cudaGetErrorString(e));
    }
    unsigned char* base = static_cast<unsigned char*>(vis);
    p.d_bucket_offset = static_cast<int64_t*>(bo);
    p.d_tile_begin = static_cast<int64_t*>(tb);
    p.d_items = static_cast<PackItem*>(it);
    p.d_vis = vis;
    p.d_vis_sq = reinterpret_cast<double*>(base + L.sq);
    p.d_vis_nf = reinterpret_cast<int32_t*>(base + L.nf);
    p.d_vis_bucket = reinterpret_cast<int32_t*>(base + L.bucket);
    p.d_vis_count = reinterpret_cast<int32_t*>(base + L.count);
    p.d_clip = clip;
    p.d_bucket_sq64 = static_cast<double*>(clip);
    p.d_clip_coef = reinterpret_cast<float*>(static_cast<unsigned char*>(clip) + clip_sq_bytes);
    p.d_status = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(clip) + clip_sq_bytes + 128);
    p.d_debug = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(clip) +
                                                      clip_sq_bytes + 192);
    p.d_chunk = chunk;
    p.d_tile_span = static_cast<int64_t*>(chunk);
    p.d_chunk_sq = reinterpret_cast<double*>(static_cast<unsigned char*>(chunk) + tb_bytes);
    p.d_chunk_nf = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(chunk) + tb_bytes + csq_bytes);
    p.seg_first = std::move(seg_first);
    p.n_seg = int32_t(seg_bucket.size());
    p.d_seg = seg;
    p.d_seg_first = reinterpret_cast<int32_t*>(sbase);
    p.d_seg_bucket = reinterpret_cast<int32_t*>(sbase + sf_bytes);
    p.d_seg_sq = reinterpret_cast<double*>(sbase + sf_bytes + sb_bytes);
    p.d_seg_nf = reinterpret_cast<long long*>(sbase + sf_bytes + sb_bytes + ss_bytes);
    p.d_bucket_done = reinterpret_cast<int32_t*>(sbase + sf_bytes + sb_bytes + ss_bytes + sn_bytes);
    p.short_first = std::move(short_first);
    p.long_first = std::move(long_first);
    p.d_short_bucket = reinterpret_cast<int32_t*>(shb);
    p.d_long_seg = reinterpret_cast<int32_t*>(shb + shb_bytes);
    p.cap_visits = cap_visits;
    p.cap_ctas = int32_t(cap_ctas);
    p.device = dev;
    return DPG_OK;
}

void release_device(Plan& p) {
    std::lock_guard<std::mutex> g(p.mu);
    if (p.device < 0) return;
    int cur = -1;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    if (cudaSetDevice(p.device) == cudaSuccess) {
        cudaFree(p.d_bucket_offset);
        cudaFree(p.d_tile_begin);
        cudaFree(p.d_items);
        cudaFree(p.d_vis);
        cudaFree(p.d_clip);
        cudaFree(p.d_chunk);
        cudaFree(p.d_seg);
    }
    if (have_cur) cudaSetDevice(cur);
    cudaGetLastError();
    p.device = -1;
}

// fp32 Adam constants, each computed in double and rounded once
int adam_constants(const dpg_hparams* hp, RsAdamArgs& a) {
    if (!hp) return fail(DPG_ERR_INVALID_ARG, "hparams is NULL");
    if (hp->step < 1) return fail(DPG_ERR_INVALID_ARG, "hparams.step must be >= 1 (got %lld)", (long long)hp->step);
    if (!(hp->beta1 >= 0.0 && hp->beta1 < 1.0) || !(hp->beta2 >= 0.0 && hp->beta2 < 1.0))
        return fail(DPG_ERR_INVALID_ARG, "betas must lie in [0, 1)");
    const double t = double(hp->step);
    a.beta1 = float(hp->beta1);
    a.beta2 = float(hp->beta2);
    a.omb1 = float(1.0 - hp->beta1);
    a.omb2 = float(1.0 - hp->beta2);
    a.bias1 = float(1.0 - std::pow(hp->beta1, t));
    a.bias2 = float(1.0 - std::pow(hp->beta2, t));
    a.lr = float(hp->lr);
    a.eps = float(hp->eps);
    a.lr_wd = float(hp->lr * hp->weight_decay);
    a.decay = hp->weight_decay != 0.0;
    return DPG_OK;
}

// fp32(1/G) with G the int64 sum of the valid-token counts
int token_scale(const int64_t* tokens, int32_t n, float* scale) {
    if (!tokens || n < 1) return fail(DPG_ERR_INVALID_ARG, "valid_tokens must hold >= 1 count");
    int64_t G = 0;
    for (int32_t k = 0; k < n; ++k) {
        if (tokens[k] < 0) return fail(DPG_ERR_INVALID_ARG, "valid_tokens[%d] < 0", k);
        if (__builtin_add_overflow(G, tokens[k], &G))
            return fail(DPG_ERR_INVALID_ARG, "valid-token sum overflows int64");
    }
    if (G == 0) return fail(DPG_ERR_ZERO_TOKENS, "global valid-token count is 0");
    *scale = float(1.0 / double(G));
    return DPG_OK;
}

}  // namespace dpg

using dpg::fail;

extern "C" {

int64_t dpg_launch_count(void) { return dpg::g_launches.load(); }

int dpg_set_fused_max_ctas(int32_t max_ctas) {
    dpg::clear_error();
    if (max_ctas < 0) return fail(DPG_ERR_INVALID_ARG, "dpg_set_fused_max_ctas: %d < 0", max_ctas);
    dpg::t_fused_max_ctas = max_ctas;
    return DPG_OK;
}

int dpg_debug_checks(const dpg_plan_t* plan, int32_t* built, int64_t* first_failure) {
    dpg::clear_error();
#ifdef DPG_DEBUG
    if (built) *built = 1;
#else
    if (built) *built = 0;
#endif
    if (first_failure) *first_failure = 0;
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_debug_checks: plan is NULL");
#ifdef DPG_DEBUG
    const dpg::Plan& p = plan->p;
    if (p.device < 0 || !first_failure) return DPG_OK;   // nothing ran on a device yet
    DPG_CUDA_TRY(cudaDeviceSynchronize());
    unsigned long long word = 0;
    DPG_CUDA_TRY(cudaMemcpy(&word, p.d_debug, sizeof word, cudaMemcpyDeviceToHost));
    DPG_CUDA_TRY(cudaMemset(p.d_debug, 0, sizeof word));
    *first_failure = static_cast<int64_t>(word);
#endif
    return DPG_OK;
}

int dpg_debug_set_limit(int64_t limit) {
    dpg::clear_error();
#ifdef DPG_DEBUG
    const char* on = std::getenv("DPG_TEST_HOOKS");
    if (!on || std::strcmp(on, "1") != 0)
        return fail(DPG_ERR_INVALID_ARG, "dpg_debug_set_limit: test hooks are disabled "
                                         "(set DPG_TEST_HOOKS=1 in the environment)");
    dpg::t_debug_limit = limit;
    return DPG_OK;
#else
    (void)limit;
    return fail(DPG_ERR_INVALID_ARG, "dpg_debug_set_limit: this library was built without "
                                     "index checks (build it with --debug)");
#endif
}

int dpg_set_programmatic_launch(int32_t on) {
    dpg::clear_error();
    if (on != 0 && on != 1)
        return fail(DPG_ERR_INVALID_ARG, "dpg_set_programmatic_launch: %d is not 0 or 1", on);
    dpg::t_programmatic = on;
    return DPG_OK;
}

int dpg_time_next_fused_launch(void* start_event, void* stop_event) {
    dpg::clear_error();
    if ((start_event == nullptr) != (stop_event == nullptr))
        return fail(DPG_ERR_INVALID_ARG, "dpg_time_next_fused_launch: give both events or neither");
    dpg::t_fused_start = static_cast<cudaEvent_t>(start_event);
    dpg::t_fused_stop = static_cast<cudaEvent_t>(stop_event);
    return DPG_OK;
}

int dpg_plan_upload(dpg_plan_t* plan) {
    dpg::clear_error();
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_plan_upload: plan is NULL");
    return dpg::upload(plan->p);
}

}  // extern "C"
