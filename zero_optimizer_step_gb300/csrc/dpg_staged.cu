// dpg_staged.cu -- the staged variant of the fused pass: a producer warp per
// CTA copies each unit's replica gradients and state into a shared-memory
// ring with the bulk-copy engine (cp.async.bulk, completion counted in bytes
// on mbarriers); every device-side wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "dpg_host.h"

namespace dpg {

constexpr uint64_t kStagedTimeoutNs = 1000000000ull;   // 1 s per wait

// ---------------------------------------------------------------------------
// Staged variant of the fused pass: the R gradient slices and the master/m/v
// slices of a unit (a tile or half of one, by R) are copied into shared memory by
// the bulk-copy engine (cp.async.bulk, completion counted in bytes on an
// mbarrier), S units ahead of the threads that consume them.  Every wait is
// bounded by a global-timer deadline: a wait that runs out records
// DPG_ERR_DEVICE_TIMEOUT in a status word, the CTA waits (again bounded) for
// its own copies still in flight and returns.  bf16 gradients, R in {1,2,4,8}.
// ---------------------------------------------------------------------------
// A unit (one ring stage) is half a tile for R = 8 and a whole tile for
// R <= 4, so that a stage holds 40-64 KB and its consumers -- one thread per
// 8-element vector -- have enough warps for the Adam arithmetic of a unit
// within the time its bytes take to stream in.
constexpr int kMaxStages = 8;
constexpr size_t kStagedSmemBudget = 200 * 1024;

__host__ __device__ constexpr int staged_unit(int R) { return R >= 8 ? kTile / 2 : kTile; }
__host__ __device__ constexpr int staged_consumers(int R) { return staged_unit(R) / kVec; }
__host__ __device__ constexpr size_t staged_stage_bytes(int R) { return size_t(staged_unit(R)) * (2 * R + 12); }
__host__ __device__ constexpr int staged_stages(int R) {
    return int(kStagedSmemBudget / staged_stage_bytes(R)) < kMaxStages
               ? int(kStagedSmemBudget / staged_stage_bytes(R)) : kMaxStages;
}

struct StagedArgs {
    RsAdamArgs a;            // buffers, tables, constants, norm scratch
    int32_t* status;         // device status word (0 = OK)
    int64_t skip_unit;       // test-only: this unit is never fetched (-1: none)
    uint64_t timeout_ns;     // bound of every wait
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 " selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0;
}
// true once the phase of `parity` completed, false if the absolute deadline
// passed first
__device__ __forceinline__ bool mbar_wait_until(uint32_t bar, uint32_t parity, uint64_t deadline) {
    while (!mbar_try_wait(bar, parity))
        if (global_ns() > deadline) return false;
    return true;
}
// the same with a relative bound, started only if the first poll fails (the
// common case -- the stage has already landed -- reads no timer)
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_until(bar, parity, global_ns() + timeout_ns);
}

// The current bucket's table entries, reloaded only when a unit leaves it.
struct BucketCursor {
    int b;
    int64_t tb_lo = 0, tb_hi = -1, bo_lo = 0, bo_hi = 0;
};

// element range [start, start + count) of unit u of U elements (count may be
// 0: the second half of a partial tile); the cursor is advanced to the
// unit's bucket
template <int U>
__device__ __forceinline__ int64_t unit_range(const RsAdamArgs& a, int64_t u, BucketCursor& c,
                                              int64_t* count) {
    constexpr int UPT = kTile / U;
    const int64_t t = u / UPT;
    if (t >= c.tb_hi) {
        c.b = bucket_of_tile(a.tile_begin, c.b, a.b1, t);
        c.tb_lo = __ldg(a.tile_begin + c.b);
        c.tb_hi = __ldg(a.tile_begin + c.b + 1);
        c.bo_lo = __ldg(a.bucket_offset + c.b);
        c.bo_hi = __ldg(a.bucket_offset + c.b + 1);
    }
    const int64_t start = c.bo_lo + (t - c.tb_lo) * kTile + (u % UPT) * U;
    const int64_t n = c.bo_hi - start;
    *count = n <= 0 ? 0 : (n < U ? n : U);
    return start;
}

template <int RT>
__device__ __forceinline__ void issue_unit(const StagedArgs& sa, unsigned char* stage, uint32_t bar,
                                           int64_t start, int64_t count) {
    constexpr int kUnit = staged_unit(RT);
    const RsAdamArgs& a = sa.a;
    const uint32_t gbytes = uint32_t(count) * 2, sbytes = uint32_t(count) * 4;
    uint64_t state;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
                 : "=l"(state) : "r"(bar), "r"(RT * gbytes + 3 * sbytes) : "memory");
    (void)state;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (count == 0) return;
#pragma unroll
    for (int r = 0; r < RT; ++r)
        asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     :: "r"(smem_u32(stage + size_t(r) * kUnit * 2)),
                        "l"(static_cast<const uint16_t*>(a.grads[r]) + start), "r"(gbytes), "r"(bar)
                     : "memory");
    const float* src[3] = {a.master, a.m, a.v};
#pragma unroll
    for (int k = 0; k < 3; ++k)
        asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     :: "r"(smem_u32(stage + size_t(RT) * kUnit * 2 + size_t(k) * kUnit * 4)),
                        "l"(src[k] + start), "r"(sbytes), "r"(bar)
                     : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    uint64_t state;
    asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];" : "=l"(state) : "r"(bar) : "memory");
    (void)state;
}

// flush_visit for a CTA with fewer warps than the kWarps partial slots per
// visit that k_norm_finalize adds up: the slots of absent warps get zeros.
template <int kConsumerWarps>
__device__ __forceinline__ void flush_visit_staged(const RsAdamArgs& a, int bucket, int visit,
                                                   double sq, int nf) {
    flush_visit(a, bucket, visit, sq, nf);
    const int64_t slot = int64_t(blockIdx.x) * a.vmax + visit;
    if ((threadIdx.x & 31) == 0)
        for (int w2 = (threadIdx.x >> 5) + kConsumerWarps; w2 < kWarps; w2 += kConsumerWarps) {
            a.vis_sq[slot * kWarps + w2] = 0.0;
            a.vis_nf[slot * kWarps + w2] = 0;
        }
}

// Warp-specialised: the consumer warps (8 for R = 8, 16 for R <= 4; one
// thread per 8-element vector of the unit) compute, the last warp produces.
// full[s] completes when stage s's copies have landed (the producer arms it
// with the byte count); empty[s] completes when every consumer warp has
// finished reading it, and the producer refills it only then.  All waits are
// bounded.
template <int RT>
__global__ void __launch_bounds__(staged_consumers(RT) + 32, 1) k_rs_adam_staged(const __grid_constant__ StagedArgs sa) {
    constexpr int S = staged_stages(RT);
    constexpr size_t SB = staged_stage_bytes(RT);
    constexpr int kUnit = staged_unit(RT);
    constexpr int kStagedThreads = staged_consumers(RT);
    constexpr int kConsumerWarps = kStagedThreads / 32;
    constexpr int UPT = kTile / kUnit;
    static_assert(kStagedThreads * kVec == kUnit, "one 8-element vector per consumer thread");
    static_assert(kConsumerWarps <= kWarps, "norm partial slots per visit");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ __align__(8) uint64_t empty[kMaxStages];
    const RsAdamArgs& a = sa.a;
    const int64_t u0 = UPT * a.t0, u1 = UPT * a.t1;   // units of the launch
    const int64_t n_mine = blockIdx.x < u1 - u0 ? (u1 - u0 - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    if (threadIdx.x == 0) {
        for (int k = 0; k < S; ++k) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(smem_u32(&full[k])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                         :: "r"(smem_u32(&empty[k])), "r"(kConsumerWarps) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (threadIdx.x >= kStagedThreads) {
        // ---------------- producer warp: one lane issues ----------------
        if (threadIdx.x != kStagedThreads) return;
        BucketCursor cur_p{a.b0};
        uint32_t armed = 0, armed_par = 0;   // stages armed at least once, parity of the last arm
        bool aborted = false;
        for (int64_t k = 0; k < n_mine; ++k) {
            const int s = int(k % S);
            if (k >= S &&
                !mbar_wait_bounded(smem_u32(&empty[s]), uint32_t((k / S - 1) & 1), sa.timeout_ns)) {
                aborted = true;
                break;
            }
            const int64_t u = u0 + blockIdx.x + k * gridDim.x;
            int64_t cnt;
            const int64_t st = unit_range<kUnit>(a, u, cur_p, &cnt);
            if (u == sa.skip_unit) continue;          // test hook: never fetched
            issue_unit<RT>(sa, smem + s * SB, smem_u32(&full[s]), st, cnt);
            armed |= 1u << s;
            armed_par = (armed_par & ~(1u << s)) | (uint32_t((k / S) & 1) << s);
        }
        if (aborted) atomicExch(sa.status, DPG_ERR_DEVICE_TIMEOUT);
        // no copy may still be in flight when this CTA exits: wait (bounded)
        // until the last phase armed on every stage has landed
        const uint64_t drain = global_ns() + sa.timeout_ns;
        for (int s2 = 0; s2 < S; ++s2)
            if (armed & (1u << s2))
                mbar_wait_until(smem_u32(&full[s2]), (armed_par >> s2) & 1u, drain);
        return;
    }

    // ---------------- consumer warps ----------------
    const int lane = threadIdx.x & 31;
    const bool norm = a.vis_sq != nullptr;
    BucketCursor cur_c{a.b0};
    int cur = -1, visit = 0;
    double sq = 0.0;
    int nf = 0;
    bool aborted = false;
    const int e = threadIdx.x * kVec;
    for (int64_t k = 0; k < n_mine; ++k) {
        const int s = int(k % S);
        const uint32_t parity = uint32_t((k / S) & 1);
        const int64_t u = u0 + blockIdx.x + k * gridDim.x;
        int64_t cnt;
        const int64_t start = unit_range<kUnit>(a, u, cur_c, &cnt);
        bool ok = mbar_wait_bounded(smem_u32(&full[s]), parity, sa.timeout_ns);
        ok = __all_sync(0xFFFFFFFFu, ok);     // warp-uniform decision
        if (!ok) {
            aborted = true;
            break;
        }
        if (norm && cur_c.b != cur) {
            if (cur >= 0) flush_visit_staged<kConsumerWarps>(a, cur, visit++, sq, nf);
            cur = cur_c.b;
            sq = 0.0;
            nf = 0;
        }
        const bool mine = e < cnt;             // counts are whole 8-element vectors
        float x[8];
        F8 w, m, v;
        if (mine) {
            const unsigned char* stage = smem + s * SB;
            widen8(*reinterpret_cast<const uint4*>(stage + size_t(e) * 2), x);
#pragma unroll
            for (int r = 1; r < RT; ++r) {
                float y[8];
                widen8(*reinterpret_cast<const uint4*>(stage + size_t(r) * kUnit * 2 + size_t(e) * 2), y);
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] = __fadd_rn(x[j], y[j]);
            }
            const float* sw = reinterpret_cast<const float*>(stage + size_t(RT) * kUnit * 2);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float4 w4 = *reinterpret_cast<const float4*>(sw + e + 4 * h);
                const float4 m4 = *reinterpret_cast<const float4*>(sw + kUnit + e + 4 * h);
                const float4 v4 = *reinterpret_cast<const float4*>(sw + 2 * kUnit + e + 4 * h);
                w.v[4 * h] = w4.x; w.v[4 * h + 1] = w4.y; w.v[4 * h + 2] = w4.z; w.v[4 * h + 3] = w4.w;
                m.v[4 * h] = m4.x; m.v[4 * h + 1] = m4.y; m.v[4 * h + 2] = m4.z; m.v[4 * h + 3] = m4.w;
                v.v[4 * h] = v4.x; v.v[4 * h + 1] = v4.y; v.v[4 * h + 2] = v4.z; v.v[4 * h + 3] = v4.w;
            }
        }
        // the warp has read stage s: release it to the producer, then compute
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        if (mine) {
            float tsq = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float g = __fmul_rn(x[j], a.scale);
                float wj = w.v[j];
                if (a.decay) wj = __fsub_rn(wj, __fmul_rn(a.lr_wd, wj));
                const float mj = __fadd_rn(__fmul_rn(a.beta1, m.v[j]), __fmul_rn(a.omb1, g));
                const float vj =
                    __fadd_rn(__fmul_rn(a.beta2, v.v[j]), __fmul_rn(a.omb2, __fmul_rn(g, g)));
                const float m_hat = __fdiv_rn(mj, a.bias1);
                const float v_hat = __fdiv_rn(vj, a.bias2);
                const float uu = __fdiv_rn(m_hat, __fadd_rn(__fsqrt_rn(v_hat), a.eps));
                w.v[j] = __fsub_rn(wj, __fmul_rn(a.lr, uu));
                m.v[j] = mj;
                v.v[j] = vj;
                tsq = fmaf(g, g, tsq);
                nf += (__float_as_uint(g) & 0x7F800000u) == 0x7F800000u;
            }
            if (norm) sq += double(tsq);
            const int64_t i = start + e;
            st_f8(a.master + i, w);
            st_f8(a.m + i, m);
            st_f8(a.v + i, v);
            const uint4 pk = narrow8(w.v);
            for (int kv = 0; kv < a.n_views; ++kv) st_u4(static_cast<uint16_t*>(a.views[kv]) + i, pk);
        }
    }
    if (aborted && lane == 0) atomicExch(sa.status, DPG_ERR_DEVICE_TIMEOUT);
    if (norm) {
        if (cur >= 0) flush_visit_staged<kConsumerWarps>(a, cur, visit++, sq, nf);
        if (threadIdx.x == 0) a.vis_count[blockIdx.x] = visit;
    }
}

// Whole step through the staged (bulk-copy) variant of the fused pass.
template <int RT>
static int launch_staged(const StagedArgs& sa, int grid, cudaStream_t s) {
    static std::mutex mu;
    static bool attr_set = false;
    const size_t smem = size_t(staged_stages(RT)) * staged_stage_bytes(RT);
    {
        std::lock_guard<std::mutex> g(mu);
        if (!attr_set) {
            DPG_CUDA_TRY(cudaFuncSetAttribute(k_rs_adam_staged<RT>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
            attr_set = true;
        }
    }
    k_rs_adam_staged<RT><<<grid, staged_consumers(RT) + 32, smem, s>>>(sa);
    return after_launch("dpg_step_staged");
}

static int step_staged(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                       const int64_t* tokens, int32_t n_counts, const dpg_hparams* hp,
                       float* master, float* m, float* v, void* const* views, int32_t n_views,
                       float* sqnorm, int64_t* nonfinite, void* stream) {
    const char* who = "dpg_step_staged";
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "%s: plan is NULL", who);
    Plan& p = const_cast<dpg_plan_t*>(plan)->p;
    if (grads_dtype != DPG_BF16)
        return fail(DPG_ERR_INVALID_ARG, "%s: bf16 gradients only", who);
    if (p.R != 1 && p.R != 2 && p.R != 4 && p.R != 8)
        return fail(DPG_ERR_INVALID_ARG, "%s: R must be 1, 2, 4 or 8 (got %d)", who, p.R);
    StagedArgs sa{};
    RsAdamArgs& a = sa.a;
    int st = fill_step_args(p, grads, grads_dtype, nullptr, hp, tokens, n_counts, master, m, v,
                            views, n_views, a, who);
    if (st != DPG_OK) return st;
    const int64_t skip = t_staged_skip;
    const int64_t tmo = t_staged_timeout_ns;
    t_staged_skip = -1;
    t_staged_timeout_ns = 0;
    if (p.n_buckets == 0) return DPG_OK;
    st = upload(p);
    if (st != DPG_OK) return st;
    a.bucket_offset = p.d_bucket_offset;
    a.tile_begin = p.d_tile_begin;
    a.t0 = 0;
    a.t1 = p.n_tiles;
    a.b0 = 0;
    a.b1 = p.n_buckets;
    int sms = 0;
    st = sm_count(p.device, &sms);
    if (st != DPG_OK) return st;
    const int64_t units = int64_t(kTile / staged_unit(p.R)) * p.n_tiles;
    const int grid = int(units < sms ? (units > 0 ? units : 1) : sms);
    const int64_t per_cta = (units + grid - 1) / grid;
    a.vmax = int32_t(per_cta < p.n_buckets ? per_cta : p.n_buckets);
    const bool want_norm = sqnorm || nonfinite;
    if (want_norm) {
        if (grid > p.cap_ctas || int64_t(grid) * a.vmax > p.cap_visits)
            return fail(DPG_ERR_CUDA, "%s: norm scratch too small", who);
        a.vis_sq = p.d_vis_sq;
        a.vis_nf = p.d_vis_nf;
        a.vis_bucket = p.d_vis_bucket;
        a.vis_count = p.d_vis_count;
    }
    sa.status = p.d_status;
    sa.skip_unit = skip;
    sa.timeout_ns = tmo > 0 ? uint64_t(tmo) : kStagedTimeoutNs;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DPG_CUDA_TRY(cudaMemsetAsync(p.d_status, 0, sizeof(int32_t), s));
    if (units > 0) {
        cudaEvent_t ev0 = t_fused_start, ev1 = t_fused_stop;
        t_fused_start = t_fused_stop = nullptr;
        if (ev0) DPG_CUDA_TRY(cudaEventRecord(ev0, s));
        switch (p.R) {
            case 1: st = launch_staged<1>(sa, grid, s); break;
            case 2: st = launch_staged<2>(sa, grid, s); break;
            case 4: st = launch_staged<4>(sa, grid, s); break;
            default: st = launch_staged<8>(sa, grid, s); break;
        }
        if (st != DPG_OK) return st;
        if (ev1) DPG_CUDA_TRY(cudaEventRecord(ev1, s));
    }
    if (want_norm) {
        st = launch_norm_finalize(a, units > 0 ? grid : 0, p.n_buckets, sqnorm, nonfinite, s,
                                  who);
    }
    return st;
}

}  // namespace dpg

using dpg::fail;

extern "C" {

int dpg_step_staged(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                    const int64_t* valid_tokens, int32_t n_counts, const dpg_hparams* hp,
                    float* master, float* exp_avg, float* exp_avg_sq, void* const* param_views,
                    int32_t n_views, float* bucket_sqnorm, int64_t* bucket_nonfinite,
                    void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_step_staged");
    return dpg::step_staged(plan, grads, grads_dtype, valid_tokens, n_counts, hp, master, exp_avg,
                            exp_avg_sq, param_views, n_views, bucket_sqnorm, bucket_nonfinite,
                            stream);
}

int dpg_check_device_status(const dpg_plan_t* plan, void* stream) {
    dpg::clear_error();
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_check_device_status: plan is NULL");
    const dpg::Plan& p = plan->p;
    if (p.device < 0) return DPG_OK;   // nothing ran on a device yet
    DPG_CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    int32_t word = 0;
    DPG_CUDA_TRY(cudaMemcpy(&word, p.d_status, sizeof word, cudaMemcpyDeviceToHost));
    if (word != 0)
        return fail(word, "dpg_check_device_status: a bounded device-side wait of the last staged "
                          "step ran out; its results are incomplete");
    return DPG_OK;
}

int dpg_set_staged_fault(int64_t skip_unit, int64_t timeout_ns) {
    dpg::clear_error();
    // a test hook: honoured only in a process that opted in through the
    // environment, so a production caller cannot arm it by accident
    const char* on = std::getenv("DPG_TEST_HOOKS");
    if (!on || std::strcmp(on, "1") != 0)
        return fail(DPG_ERR_INVALID_ARG, "dpg_set_staged_fault: test hooks are disabled "
                                         "(set DPG_TEST_HOOKS=1 in the environment)");
    dpg::t_staged_skip = skip_unit;
    dpg::t_staged_timeout_ns = timeout_ns;
    return DPG_OK;
}

}  // extern "C"
