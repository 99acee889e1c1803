// dpg_kernels.cu -- sm_103a kernels and the device half of the libdpg C ABI.
//
// Everything on this path is a stream of HBM traffic with a few dozen ALU
// operations per element, so the kernels are built for bandwidth:
//   * one thread owns one 8-element vector: 128-bit loads of every bf16
//     replica gradient, 256-bit loads/stores of the fp32 master/m/v state;
//   * persistent grids (SM count x resident CTAs) striding over bucket-aligned
//     tiles, so the whole GPU streams through the flat buffers in one wave;
//   * the reduce-scatter, the normalisation, Adam and the bf16 all-gather are
//     ONE pass: every byte of the step is read or written exactly once;
//   * per-bucket squared-norm partials are warp-shuffle reductions written per
//     (tile, warp) and summed in a fixed order by a small second kernel, so
//     the norms are deterministic run to run.
// Arithmetic of the update uses the IEEE round-to-nearest intrinsics
// (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn, __fsub_rn), which the compiler
// never contracts into FMAs, in the order of Kingma & Ba's Algorithm 1.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "dpg_internal.h"

namespace dpg {

static std::atomic<int64_t> g_launches{0};
static thread_local cudaEvent_t t_fused_start = nullptr, t_fused_stop = nullptr;
// test-only fault injection of the staged pass (consumed by its next launch)
static thread_local int64_t t_staged_skip = -1;
// Upper bound on the CTAs of the fused passes launched from this thread
// (0: one per SM, the default).  A smaller grid leaves SMs to concurrent work.
static thread_local int32_t t_fused_max_ctas = 0;
static thread_local int64_t t_staged_timeout_ns = 0;
constexpr uint64_t kStagedTimeoutNs = 1000000000ull;   // 1 s per wait

#define DPG_CUDA_TRY(call)                                                              \
    do {                                                                                \
        cudaError_t e_ = (call);                                                        \
        if (e_ != cudaSuccess)                                                          \
            return fail(DPG_ERR_CUDA, "%s: %s (%s)", __func__, cudaGetErrorString(e_),  \
                        #call);                                                         \
    } while (0)

// ---------------------------------------------------------------------------
// memory access: streaming vector loads and stores (inline PTX)
// ---------------------------------------------------------------------------
struct F8 {
    float v[8];
};

// read-only gradient stream: bypass L1 (an L2 evict-first hint measured 0.4 % slower)
__device__ __forceinline__ uint4 ld_grad_u4(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ F8 ld_grad_f8(const float* p) {
    F8 r;
    asm("ld.global.nc.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]), "=f"(r.v[5]),
          "=f"(r.v[6]), "=f"(r.v[7])
        : "l"(p));
    return r;
}

// read-modify-write state (master / m / v / accumulation buffer)
__device__ __forceinline__ F8 ld_state_f8(const float* p) {
    F8 r;
    asm("ld.global.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]), "=f"(r.v[5]),
          "=f"(r.v[6]), "=f"(r.v[7])
        : "l"(p));
    return r;
}

__device__ __forceinline__ void st_f8(float* p, const F8& x) {
    asm volatile("st.global.L1::no_allocate.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
                 "f"(x.v[0]), "f"(x.v[1]), "f"(x.v[2]), "f"(x.v[3]), "f"(x.v[4]), "f"(x.v[5]),
                 "f"(x.v[6]), "f"(x.v[7]));
}

__device__ __forceinline__ void st_u4(void* p, uint4 x) {
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(x.x),
                 "r"(x.y), "r"(x.z), "r"(x.w));
}

// bf16 pair (low half = lower address) -> two exact fp32 values
__device__ __forceinline__ void widen2(uint32_t u, float& lo, float& hi) {
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xFFFF0000u);
}

__device__ __forceinline__ void widen8(uint4 x, float* f) {
    widen2(x.x, f[0], f[1]);
    widen2(x.y, f[2], f[3]);
    widen2(x.z, f[4], f[5]);
    widen2(x.w, f[6], f[7]);
}

// eight fp32 -> eight bf16 (round to nearest even), packed for a 128-bit store
__device__ __forceinline__ uint4 narrow8(const float* f) {
    uint4 r;
    __nv_bfloat162 h;
    h = __floats2bfloat162_rn(f[0], f[1]);
    r.x = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(f[2], f[3]);
    r.y = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(f[4], f[5]);
    r.z = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(f[6], f[7]);
    r.w = *reinterpret_cast<uint32_t*>(&h);
    return r;
}

// ---------------------------------------------------------------------------
// fused reduce-scatter -> scale -> Adam -> all-gather
// ---------------------------------------------------------------------------
// kInF32PlusBf16x2: fp32 accumulation buffers plus the last TWO bf16
// microbatches, folded in microbatch order.
enum : int { kInBf16 = 0, kInF32 = 1, kInF32PlusBf16 = 2, kInReduced = 3, kInF32PlusBf16x2 = 4 };

// Passes of the fused kernel.  kFull: reduce, scale, Adam, cast (the step).
// With global norm clipping the step takes two passes: the norm pass
// (k_norm_pass) reduces, scales, sums the squares and may store g; kUpdate
// then multiplies g by the clip coefficient found on the device and runs Adam.
enum : int { kFull = 0, kNormOnly = 1, kUpdate = 2 };

struct RsAdamArgs {
    const void* grads[DPG_MAX_REPLICAS];
    const void* last[DPG_MAX_REPLICAS];
    const void* last2[DPG_MAX_REPLICAS];  // kInF32PlusBf16x2: the final microbatch
    void* views[DPG_MAX_VIEWS];
    float* master;
    float* m;
    float* v;
    float* reduced;      // nullable
    double* vis_sq;      // per-(CTA, bucket visit, warp) norm partials; NULL: no norm
    int32_t* vis_nf;     // same layout, non-finite counts
    int32_t* vis_bucket; // bucket of each (CTA, visit)
    int32_t* vis_count;  // visits made by each CTA
    int32_t vmax;        // visit slots per CTA
    const int64_t* bucket_offset;
    const int64_t* tile_begin;
    int64_t t0, t1;      // tile range of buckets [b0, b1)
    int32_t b0, b1;
    int32_t R, n_views;
    float scale;         // fp32(1/G)
    float beta1, beta2, omb1, omb2, bias1, bias2, lr, eps, lr_wd;
    int32_t decay;
    const float* g_in;      // kInReduced: the normalised reduced gradient
    const float* clip_coef; // kUpdate: device scalar, g <- g * coef
    // chunked launches (one CTA per chunk): tile -> bucket map and the
    // per-chunk norm partials (NULL: no norm)
    const int32_t* tile_bucket;
    double* chunk_sq;
    int32_t* chunk_nf;
};

// Bucket holding tile t, searching forward from bucket b (tile_begin[b] <= t
// and t < tile_begin[b_end] hold on entry).  Empty buckets are skipped.
__device__ __forceinline__ int bucket_of_tile(const int64_t* tile_begin, int b, int b_end,
                                              int64_t t) {
    if (t < __ldg(tile_begin + b + 1)) return b;
    int lo = b + 1, hi = b_end;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(tile_begin + mid) <= t) lo = mid;
        else hi = mid;
    }
    return lo;
}

// x_r widened (and, for the accumulation path, plus the last microbatch),
// summed in rank order 0..R-1 in binary32.
template <int RT, int MODE>
__device__ __forceinline__ void reduce_vector(const RsAdamArgs& a, int64_t i, float* s) {
    const int R = RT > 0 ? RT : a.R;
    if constexpr (MODE == kInReduced) {
        const F8 x = ld_grad_f8(a.g_in + i);
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j] = x.v[j];
    } else if constexpr (MODE == kInBf16) {
        if constexpr (RT > 0) {
            uint4 x[RT];
#pragma unroll
            for (int r = 0; r < RT; ++r)
                x[r] = ld_grad_u4(static_cast<const uint16_t*>(a.grads[r]) + i);
            widen8(x[0], s);
#pragma unroll
            for (int r = 1; r < RT; ++r) {
                float t[8];
                widen8(x[r], t);
#pragma unroll
                for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], t[j]);
            }
        } else {
            widen8(ld_grad_u4(static_cast<const uint16_t*>(a.grads[0]) + i), s);
#pragma unroll 4
            for (int r = 1; r < R; ++r) {
                float t[8];
                widen8(ld_grad_u4(static_cast<const uint16_t*>(a.grads[r]) + i), t);
#pragma unroll
                for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], t[j]);
            }
        }
    } else {
        // fp32 accumulation buffers (optionally + the final bf16 microbatch)
#pragma unroll(RT > 0 ? RT : 2)
        for (int r = 0; r < R; ++r) {
            F8 x = ld_grad_f8(static_cast<const float*>(a.grads[r]) + i);
            if constexpr (MODE == kInF32PlusBf16 || MODE == kInF32PlusBf16x2) {
                float t[8];
                widen8(ld_grad_u4(static_cast<const uint16_t*>(a.last[r]) + i), t);
#pragma unroll
                for (int j = 0; j < 8; ++j) x.v[j] = __fadd_rn(x.v[j], t[j]);
            }
            if constexpr (MODE == kInF32PlusBf16x2) {
                float t[8];
                widen8(ld_grad_u4(static_cast<const uint16_t*>(a.last2[r]) + i), t);
#pragma unroll
                for (int j = 0; j < 8; ++j) x.v[j] = __fadd_rn(x.v[j], t[j]);
            }
            if (r == 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j) s[j] = x.v[j];
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], x.v[j]);
            }
        }
    }
}

// Per-bucket norm bookkeeping: a CTA's consecutive tiles of one bucket form a
// "visit"; each thread keeps running sums over the visit (per-tile fp32 sums
// of 8 squares, accumulated in double), and the warps reduce and store them
// only when the CTA moves on to the next bucket -- once or twice per CTA for
// large buckets, so no shuffle or store sits on the per-tile critical path.
__device__ __forceinline__ void flush_visit(const RsAdamArgs& a, int bucket, int visit, double sq,
                                            int nf) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
        nf += __shfl_xor_sync(0xFFFFFFFFu, nf, o);
    }
    const int64_t slot = int64_t(blockIdx.x) * a.vmax + visit;
    if (lane == 0) {
        a.vis_sq[slot * kWarps + warp] = sq;
        a.vis_nf[slot * kWarps + warp] = nf;
    }
    if (threadIdx.x == 0) a.vis_bucket[slot] = bucket;
}

template <int RT, int MODE, int PHASE>
__global__ void __launch_bounds__(kThreads, 1) k_rs_adam(const __grid_constant__ RsAdamArgs a) {
    static_assert(PHASE != kNormOnly, "the norm pass is k_norm_pass");
    const bool norm = PHASE != kUpdate && a.vis_sq != nullptr;
    float coef = 1.0f;
    if constexpr (PHASE == kUpdate) coef = __ldg(a.clip_coef);
    int b = a.b0;
    int cur = -1;  // bucket of the running norm sums
    int visit = 0;
    double sq = 0.0;
    int nf = 0;
    // the current bucket's table entries, reloaded only when a tile leaves it
    // (per-tile lookups were half of the load requests of the lighter passes)
    int64_t tb_lo = 0, tb_hi = -1, bo_lo = 0, bo_hi = 0;
    for (int64_t t = a.t0 + blockIdx.x; t < a.t1; t += gridDim.x) {
        if (t >= tb_hi) {                                   // CTA-uniform
            b = bucket_of_tile(a.tile_begin, b, a.b1, t);
            tb_lo = __ldg(a.tile_begin + b);
            tb_hi = __ldg(a.tile_begin + b + 1);
            bo_lo = __ldg(a.bucket_offset + b);
            bo_hi = __ldg(a.bucket_offset + b + 1);
        }
        if (norm && b != cur) {
            if (cur >= 0) flush_visit(a, cur, visit++, sq, nf);
            cur = b;
            sq = 0.0;
            nf = 0;
        }
        const int64_t bucket_end = bo_hi;
        const int64_t i = bo_lo + (t - tb_lo) * kTile + int64_t(threadIdx.x) * kVec;
        if (i < bucket_end) {
            float s[8];
            reduce_vector<RT, MODE>(a, i, s);
            float g[8];
            {
                F8 w = ld_state_f8(a.master + i);
                F8 m = ld_state_f8(a.m + i);
                F8 v = ld_state_f8(a.v + i);
                float tsq = 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    g[j] = MODE == kInReduced ? s[j] : __fmul_rn(s[j], a.scale);
                    if constexpr (PHASE == kUpdate) g[j] = __fmul_rn(g[j], coef);
                    float wj = w.v[j];
                    if (a.decay) wj = __fsub_rn(wj, __fmul_rn(a.lr_wd, wj));
                    const float mj = __fadd_rn(__fmul_rn(a.beta1, m.v[j]), __fmul_rn(a.omb1, g[j]));
                    const float vj = __fadd_rn(__fmul_rn(a.beta2, v.v[j]),
                                               __fmul_rn(a.omb2, __fmul_rn(g[j], g[j])));
                    const float m_hat = __fdiv_rn(mj, a.bias1);
                    const float v_hat = __fdiv_rn(vj, a.bias2);
                    const float u = __fdiv_rn(m_hat, __fadd_rn(__fsqrt_rn(v_hat), a.eps));
                    w.v[j] = __fsub_rn(wj, __fmul_rn(a.lr, u));
                    m.v[j] = mj;
                    v.v[j] = vj;
                    tsq = fmaf(g[j], g[j], tsq);
                    nf += (__float_as_uint(g[j]) & 0x7F800000u) == 0x7F800000u;
                }
                if (norm) sq += double(tsq);
                st_f8(a.master + i, w);
                st_f8(a.m + i, m);
                st_f8(a.v + i, v);
                const uint4 p = narrow8(w.v);
                for (int k = 0; k < a.n_views; ++k) st_u4(static_cast<uint16_t*>(a.views[k]) + i, p);
                if (PHASE == kFull && a.reduced) {
                    F8 gg;
#pragma unroll
                    for (int j = 0; j < 8; ++j) gg.v[j] = g[j];
                    st_f8(a.reduced + i, gg);
                }
            }
        }
    }
    if (norm) {
        if (cur >= 0) flush_visit(a, cur, visit++, sq, nf);
        if (threadIdx.x == 0) a.vis_count[blockIdx.x] = visit;
    }
}

// ---------------------------------------------------------------------------
// Norm pass of the clipped step: reduce, scale, squares per bucket visit, and
// optionally store g.  It moves only 2R (+4) bytes per element, so each
// iteration handles two tiles (t and t + grid) with the loads of both in
// flight before either is summed; the tile order, and with it the visits, is
// that of the single-tile loop.
// ---------------------------------------------------------------------------
template <int RT, int MODE> struct Raw;
template <int RT> struct Raw<RT, kInBf16> { uint4 x[RT]; };
template <int RT> struct Raw<RT, kInF32> { F8 x[RT]; };
template <int RT> struct Raw<RT, kInF32PlusBf16> { F8 x[RT]; uint4 l[RT]; };

template <int RT, int MODE>
__device__ __forceinline__ void load_raw(const RsAdamArgs& a, int64_t i, Raw<RT, MODE>& raw) {
#pragma unroll
    for (int r = 0; r < RT; ++r) {
        if constexpr (MODE == kInBf16) {
            raw.x[r] = ld_grad_u4(static_cast<const uint16_t*>(a.grads[r]) + i);
        } else {
            raw.x[r] = ld_grad_f8(static_cast<const float*>(a.grads[r]) + i);
            if constexpr (MODE == kInF32PlusBf16)
                raw.l[r] = ld_grad_u4(static_cast<const uint16_t*>(a.last[r]) + i);
        }
    }
}

// the same rank-ordered binary32 sum as reduce_vector
template <int RT, int MODE>
__device__ __forceinline__ void sum_raw(const Raw<RT, MODE>& raw, float* s) {
#pragma unroll
    for (int r = 0; r < RT; ++r) {
        float x[8];
        if constexpr (MODE == kInBf16) {
            widen8(raw.x[r], x);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = raw.x[r].v[j];
            if constexpr (MODE == kInF32PlusBf16) {
                float t[8];
                widen8(raw.l[r], t);
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] = __fadd_rn(x[j], t[j]);
            }
        }
        if (r == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) s[j] = x[j];
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], x[j]);
        }
    }
}

// g = s * scale; its squares are added to a running double-float sum (hi, lo)
// with binary32 operations only -- binary64 arithmetic is scarce on this GPU,
// so the sum is widened to double once per bucket visit: p + e is g*g exactly
// (FMA) and Knuth's TwoSum keeps the rounding error of hi in lo (about 2^-48
// relative overall).  |g| >= 2^60, whose binary32 square would overflow, is
// squared in binary64 (`big`).
struct NormAcc {
    float hi = 0.0f, lo = 0.0f;
    double big = 0.0;
    __device__ double value() const { return (double(hi) + double(lo)) + big; }
};

__device__ __forceinline__ void two_sum_square(NormAcc& acc, float x) {
    const float p = __fmul_rn(x, x);
    const float e = fmaf(x, x, -p);
    const float t = __fadd_rn(acc.hi, p);
    const float bp = __fsub_rn(t, acc.hi);
    const float err = __fadd_rn(__fsub_rn(acc.hi, __fsub_rn(t, bp)), __fsub_rn(p, bp));
    acc.hi = t;
    acc.lo = __fadd_rn(acc.lo, __fadd_rn(err, e));
}

__device__ __forceinline__ void norm_vector(const RsAdamArgs& a, int64_t i, const float* s,
                                            NormAcc& acc, int& nf, bool squares) {
    float g[8];
    bool rare = false;   // a huge or non-finite value in this vector
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        g[j] = __fmul_rn(s[j], a.scale);
        rare |= !(fabsf(g[j]) < 0x1p60f);
    }
    if (!squares) {      // all-reduce only: no norm requested
        if (a.reduced) {
            F8 gg;
#pragma unroll
            for (int j = 0; j < 8; ++j) gg.v[j] = g[j];
            st_f8(a.reduced + i, gg);
        }
        return;
    }
    // a branch uniform over the active lanes (callers may be inside a partial
    // tile's per-thread condition): the binary64 path must not be if-converted
    // into predicated binary64 instructions issued for every element
    if (__any_sync(__activemask(), rare)) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (fabsf(g[j]) < 0x1p60f) two_sum_square(acc, g[j]);
            else acc.big += double(g[j]) * double(g[j]);
            nf += (__float_as_uint(g[j]) & 0x7F800000u) == 0x7F800000u;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) two_sum_square(acc, g[j]);
    }
    if (a.reduced) {
        F8 gg;
#pragma unroll
        for (int j = 0; j < 8; ++j) gg.v[j] = g[j];
        st_f8(a.reduced + i, gg);
    }
}

// tiles per iteration of the norm pass: about 64 registers of loads in flight
template <int RT, int MODE>
constexpr int norm_tiles_per_iter() {
    constexpr int regs = RT * (MODE == kInBf16 ? 4 : MODE == kInF32 ? 8 : 12);
    return RT == 0 ? 1 : (64 / regs < 1 ? 1 : (64 / regs > 4 ? 4 : 64 / regs));
}

template <int RT, int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_norm_pass(const __grid_constant__ RsAdamArgs a) {
    constexpr int TPI = norm_tiles_per_iter<RT, MODE>();
    const bool norm = a.vis_sq != nullptr;
    int b = a.b0, cur = -1, visit = 0;
    NormAcc acc;
    int nf = 0;
    int64_t tb_lo = 0, tb_hi = -1, bo_lo = 0, bo_hi = 0;
    const int64_t G = gridDim.x;
    for (int64_t t = a.t0 + blockIdx.x; t < a.t1; t += TPI * G) {
        int bu[TPI];
        int64_t iu[TPI], eu[TPI];
#pragma unroll
        for (int u = 0; u < TPI; ++u) {
            const int64_t tu = t + u * G;
            bu[u] = -1;
            iu[u] = 0;
            eu[u] = 0;
            if (tu < a.t1) {
                if (tu >= tb_hi) {                      // CTA-uniform
                    b = bucket_of_tile(a.tile_begin, b, a.b1, tu);
                    tb_lo = __ldg(a.tile_begin + b);
                    tb_hi = __ldg(a.tile_begin + b + 1);
                    bo_lo = __ldg(a.bucket_offset + b);
                    bo_hi = __ldg(a.bucket_offset + b + 1);
                }
                bu[u] = b;
                eu[u] = bo_hi;
                iu[u] = bo_lo + (tu - tb_lo) * kTile + int64_t(threadIdx.x) * kVec;
            }
        }
        if constexpr (RT > 0) {
            Raw<RT, MODE> raw[TPI];
#pragma unroll
            for (int u = 0; u < TPI; ++u)
                if (iu[u] < eu[u]) load_raw<RT, MODE>(a, iu[u], raw[u]);
#pragma unroll
            for (int u = 0; u < TPI; ++u) {
                if (bu[u] < 0) break;                   // past the end: CTA-uniform
                if (norm && bu[u] != cur) {
                    if (cur >= 0) flush_visit(a, cur, visit++, acc.value(), nf);
                    cur = bu[u];
                    acc = NormAcc();
                    nf = 0;
                }
                if (iu[u] < eu[u]) {
                    float su[8];
                    sum_raw<RT, MODE>(raw[u], su);
                    norm_vector(a, iu[u], su, acc, nf, norm);
                }
            }
        } else {
            if (norm && bu[0] != cur) {
                if (cur >= 0) flush_visit(a, cur, visit++, acc.value(), nf);
                cur = bu[0];
                acc = NormAcc();
                nf = 0;
            }
            if (iu[0] < eu[0]) {
                float su[8];
                reduce_vector<RT, MODE>(a, iu[0], su);
                norm_vector(a, iu[0], su, acc, nf, norm);
            }
        }
    }
    if (norm) {
        if (cur >= 0) flush_visit(a, cur, visit++, acc.value(), nf);
        if (threadIdx.x == 0) a.vis_count[blockIdx.x] = visit;
    }
}

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

// One CTA per bucket: thread c (and c + 256, ...) finds CTA c's visit of the
// bucket by binary search in that CTA's visit list (its buckets increase) and
// adds the visit's warp partials in warp order; the block then combines the
// threads in a fixed tree.  The order depends only on the launch geometry, so
// the norms are the same from run to run.
constexpr int kFinalizeThreads = 256;

__global__ void __launch_bounds__(kFinalizeThreads)
k_norm_finalize(const double* __restrict__ vis_sq, const int32_t* __restrict__ vis_nf,
                const int32_t* __restrict__ vis_bucket, const int32_t* __restrict__ vis_count,
                int32_t n_cta, int32_t vmax, int32_t b0, float* sqnorm, int64_t* nonfinite,
                double* sqnorm64) {
    __shared__ double s_sq[kFinalizeThreads];
    __shared__ long long s_nf[kFinalizeThreads];
    const int b = b0 + blockIdx.x;
    double acc = 0.0;
    long long cnt = 0;
    for (int c = threadIdx.x; c < n_cta; c += kFinalizeThreads) {
        const int32_t* vb = vis_bucket + int64_t(c) * vmax;
        const int n = vis_count[c];
        int lo = 0, hi = n;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (vb[mid] < b) lo = mid + 1;
            else hi = mid;
        }
        if (lo < n && vb[lo] == b) {
            const int64_t slot = (int64_t(c) * vmax + lo) * kWarps;
            for (int w = 0; w < kWarps; ++w) {
                acc += vis_sq[slot + w];
                cnt += vis_nf[slot + w];
            }
        }
    }
    s_sq[threadIdx.x] = acc;
    s_nf[threadIdx.x] = cnt;
    __syncthreads();
    for (int w = kFinalizeThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) {
            s_sq[threadIdx.x] += s_sq[threadIdx.x + w];
            s_nf[threadIdx.x] += s_nf[threadIdx.x + w];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        if (sqnorm) sqnorm[b] = float(s_sq[0]);
        if (nonfinite) nonfinite[b] = s_nf[0];
        if (sqnorm64) sqnorm64[b] = s_sq[0];
    }
}

// ---------------------------------------------------------------------------
// Chunked launch of the fused pass: one 128-thread CTA per 1024-element chunk
// (a quarter tile), one 8-element vector per thread, no grid-stride loop.  The
// SM keeps several such CTAs resident at different points of their
// load -> Adam -> store sequence, so DRAM stays busy while some of them do
// arithmetic; a persistent CTA of 16 warps that load and compute in step
// leaves it idle meanwhile.  Norms: each CTA writes one (sum of squares,
// non-finite count) partial per chunk; k_chunk_finalize adds a bucket's
// chunks in a fixed order.
// ---------------------------------------------------------------------------
constexpr int kChunkThreads = 128;
constexpr int kChunk = kChunkThreads * kVec;
constexpr int kChunksPerTile = int(kTile / kChunk);

// Adam on one 8-element vector of the chunked pass: s is the rank-ordered
// sum; adds the vector's squares and non-finite count to sq / nf.
template <int MODE, int PHASE>
__device__ __forceinline__ void adam_vector(const RsAdamArgs& a, int64_t i, const float* s,
                                            float coef, float& sq, int& nf) {
    F8 w = ld_state_f8(a.master + i);
    F8 m = ld_state_f8(a.m + i);
    F8 v = ld_state_f8(a.v + i);
    float g[8];
    float tsq = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        g[j] = MODE == kInReduced ? s[j] : __fmul_rn(s[j], a.scale);
        if constexpr (PHASE == kUpdate) g[j] = __fmul_rn(g[j], coef);
        float wj = w.v[j];
        if (a.decay) wj = __fsub_rn(wj, __fmul_rn(a.lr_wd, wj));
        const float mj = __fadd_rn(__fmul_rn(a.beta1, m.v[j]), __fmul_rn(a.omb1, g[j]));
        const float vj = __fadd_rn(__fmul_rn(a.beta2, v.v[j]),
                                   __fmul_rn(a.omb2, __fmul_rn(g[j], g[j])));
        const float m_hat = __fdiv_rn(mj, a.bias1);
        const float v_hat = __fdiv_rn(vj, a.bias2);
        const float u = __fdiv_rn(m_hat, __fadd_rn(__fsqrt_rn(v_hat), a.eps));
        w.v[j] = __fsub_rn(wj, __fmul_rn(a.lr, u));
        m.v[j] = mj;
        v.v[j] = vj;
        tsq = fmaf(g[j], g[j], tsq);
        nf += (__float_as_uint(g[j]) & 0x7F800000u) == 0x7F800000u;
    }
    sq = tsq;
    st_f8(a.master + i, w);
    st_f8(a.m + i, m);
    st_f8(a.v + i, v);
    const uint4 p = narrow8(w.v);
    for (int k = 0; k < a.n_views; ++k) st_u4(static_cast<uint16_t*>(a.views[k]) + i, p);
    if (PHASE == kFull && a.reduced) {
        F8 gg;
#pragma unroll
        for (int j = 0; j < 8; ++j) gg.v[j] = g[j];
        st_f8(a.reduced + i, gg);
    }
}

template <int RT, int MODE, int PHASE>
__global__ void __launch_bounds__(kChunkThreads) k_rs_adam_chunk(const __grid_constant__ RsAdamArgs a) {
    // kNormOnly: reduce and scale only -- g to a.reduced, norm partials, no
    // Adam (the all-reduce of the DDP schedule)
    const int64_t c = blockIdx.x;                         // chunk of this launch
    const int64_t t = a.t0 + c / kChunksPerTile;
    const int b = __ldg(a.tile_bucket + t);
    const int64_t i = __ldg(a.bucket_offset + b) + (t - __ldg(a.tile_begin + b)) * kTile +
                      (c % kChunksPerTile) * kChunk + int64_t(threadIdx.x) * kVec;
    float sq = 0.0f;
    int nf = 0;
    if (i < __ldg(a.bucket_offset + b + 1)) {
        float coef = 1.0f;
        if constexpr (PHASE == kUpdate) coef = __ldg(a.clip_coef);
        float s[8];
        reduce_vector<RT, MODE>(a, i, s);
        if constexpr (PHASE == kNormOnly) {
            F8 gg;
            float tsq = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                gg.v[j] = __fmul_rn(s[j], a.scale);
                tsq = fmaf(gg.v[j], gg.v[j], tsq);
                nf += (__float_as_uint(gg.v[j]) & 0x7F800000u) == 0x7F800000u;
            }
            sq = tsq;
            st_f8(a.reduced + i, gg);
        } else {
            adam_vector<MODE, PHASE>(a, i, s, coef, sq, nf);
        }
    }
    if (a.chunk_sq != nullptr) {                          // uniform over the launch
        // a warp's 256 squares summed in fp32 (relative error ~1e-7), the
        // CTA's four warps and the bucket's chunks in double
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
        nf = __reduce_add_sync(0xFFFFFFFFu, nf);
        __shared__ double w_sq[kChunkThreads / 32];
        __shared__ int w_nf[kChunkThreads / 32];
        if ((threadIdx.x & 31) == 0) {
            w_sq[threadIdx.x >> 5] = double(sq);
            w_nf[threadIdx.x >> 5] = nf;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            double tot = 0.0;
            int cnt = 0;
#pragma unroll
            for (int k = 0; k < kChunkThreads / 32; ++k) {
                tot += w_sq[k];
                cnt += w_nf[k];
            }
            a.chunk_sq[c] = tot;
            a.chunk_nf[c] = cnt;
        }
    }
}

// Chunked norm pass of the clipped step: reduce, scale, optionally store g,
// and sum the squares near-exactly (fp32 double-float per thread, see
// two_sum_square), one double partial per chunk.  The warps combine their
// double-float pairs with fp32 TwoSum; the rare binary64 term (huge or
// non-finite values) is combined only when some lane of the warp has one, so
// the per-element path issues no binary64 instruction.
template <int RT, int MODE, int NT>
__global__ void __launch_bounds__(NT) k_norm_chunk(const __grid_constant__ RsAdamArgs a) {
    constexpr int CH = NT * kVec;                         // elements per chunk
    constexpr int CPT = int(kTile / CH);
    static_assert(CPT >= 1 && CPT * CH == kTile, "a tile holds a whole number of chunks");
    const int64_t c = blockIdx.x;
    const int64_t t = a.t0 + c / CPT;
    const int b = __ldg(a.tile_bucket + t);
    const int64_t i = __ldg(a.bucket_offset + b) + (t - __ldg(a.tile_begin + b)) * kTile +
                      (c % CPT) * CH + int64_t(threadIdx.x) * kVec;
    const bool norm = a.chunk_sq != nullptr;
    NormAcc acc;
    int nf = 0;
    if (i < __ldg(a.bucket_offset + b + 1)) {
        float s[8];
        reduce_vector<RT, MODE>(a, i, s);
        norm_vector(a, i, s, acc, nf, norm);
    }
    if (!norm) return;                                    // uniform over the launch
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ohi = __shfl_xor_sync(0xFFFFFFFFu, acc.hi, o);
        const float olo = __shfl_xor_sync(0xFFFFFFFFu, acc.lo, o);
        const float sh = __fadd_rn(acc.hi, ohi);
        const float bp = __fsub_rn(sh, acc.hi);
        const float err = __fadd_rn(__fsub_rn(acc.hi, __fsub_rn(sh, bp)), __fsub_rn(ohi, bp));
        acc.hi = sh;
        acc.lo = __fadd_rn(__fadd_rn(acc.lo, olo), err);
    }
    if (__any_sync(0xFFFFFFFFu, acc.big != 0.0)) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc.big += __shfl_xor_sync(0xFFFFFFFFu, acc.big, o);
    }
    nf = __reduce_add_sync(0xFFFFFFFFu, nf);
    __shared__ double w_sq[NT / 32];
    __shared__ int w_nf[NT / 32];
    if ((threadIdx.x & 31) == 0) {
        w_sq[threadIdx.x >> 5] = acc.value();
        w_nf[threadIdx.x >> 5] = nf;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        int cnt = 0;
#pragma unroll
        for (int k = 0; k < NT / 32; ++k) {
            tot += w_sq[k];
            cnt += w_nf[k];
        }
        a.chunk_sq[c] = tot;
        a.chunk_nf[c] = cnt;
    }
}

// One CTA per bucket of a chunked launch starting at tile t0.  A bucket of a
// large plan has 10^5 chunk partials and there are only tens of buckets, so
// each thread keeps 8 loads in flight: thread j adds chunks j + 1024 k in
// increasing k (8 at a time, in order), then a fixed tree combines the
// threads -- the same order on every run.
constexpr int kChunkFinalizeThreads = 1024;

__global__ void __launch_bounds__(kChunkFinalizeThreads)
k_chunk_finalize(const double* __restrict__ chunk_sq, const int32_t* __restrict__ chunk_nf,
                 const int64_t* __restrict__ tile_begin, int64_t t0, int32_t cpt, int32_t b0,
                 float* sqnorm, int64_t* nonfinite, double* sqnorm64) {
    constexpr int T = kChunkFinalizeThreads, U = 8;
    __shared__ double s_sq[T];
    __shared__ long long s_nf[T];
    const int b = b0 + blockIdx.x;
    const int64_t c0 = (__ldg(tile_begin + b) - t0) * cpt;
    const int64_t c1 = (__ldg(tile_begin + b + 1) - t0) * cpt;
    double acc = 0.0;
    long long cnt = 0;
    for (int64_t c = c0 + threadIdx.x; c < c1; c += int64_t(T) * U) {
        double x[U];
        int y[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = c + int64_t(u) * T;
            x[u] = k < c1 ? chunk_sq[k] : 0.0;
            y[u] = k < c1 ? chunk_nf[k] : 0;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            acc += x[u];
            cnt += y[u];
        }
    }
    s_sq[threadIdx.x] = acc;
    s_nf[threadIdx.x] = cnt;
    __syncthreads();
    for (int w = T / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) {
            s_sq[threadIdx.x] += s_sq[threadIdx.x + w];
            s_nf[threadIdx.x] += s_nf[threadIdx.x + w];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        if (sqnorm) sqnorm[b] = float(s_sq[0]);
        if (nonfinite) nonfinite[b] = s_nf[0];
        if (sqnorm64) sqnorm64[b] = s_sq[0];
    }
}

// Global clip coefficient from the per-bucket squared norms (one CTA, fixed
// order): norm = sqrt(sum), coef = min(1, max_norm / (norm + 1e-6)) in double,
// stored as fp32; a NaN norm gives a NaN coefficient (it is not clamped away).
__global__ void __launch_bounds__(256) k_clip_coef(const double* __restrict__ bucket_sq, int32_t nb,
                                                   double max_norm, float* coef, float* out) {
    __shared__ double sh[256];
    double acc = 0.0;
    for (int b = threadIdx.x; b < nb; b += 256) acc += bucket_sq[b];
    sh[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double norm = sqrt(sh[0]);
        double c = max_norm / (norm + 1e-6);
        if (c > 1.0) c = 1.0;
        *coef = float(c);
        if (out) {
            out[0] = float(norm);
            out[1] = float(c);
        }
    }
}

// ---------------------------------------------------------------------------
// no_sync accumulation and the stand-alone all-gather
// ---------------------------------------------------------------------------
template <bool FIRST>
__global__ void __launch_bounds__(256) k_accumulate(const uint16_t* __restrict__ g,
                                                    float* __restrict__ acc, int64_t n_vec) {
    for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < n_vec;
         k += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = k * kVec;
        float x[8];
        widen8(ld_grad_u4(g + i), x);
        F8 r;
        if (FIRST) {
#pragma unroll
            for (int j = 0; j < 8; ++j) r.v[j] = x[j];
        } else {
            const F8 a = ld_state_f8(acc + i);
#pragma unroll
            for (int j = 0; j < 8; ++j) r.v[j] = __fadd_rn(a.v[j], x[j]);
        }
        st_f8(acc + i, r);
    }
}

// Two microbatches folded into the fp32 buffer in one pass, in microbatch
// order: acc <- (acc + f32(a)) + f32(b), or f32(a) + f32(b) for the first
// pair -- the same two binary32 additions as two k_accumulate launches, with
// the accumulator read and written once instead of twice.
template <bool FIRST>
__global__ void __launch_bounds__(256) k_accumulate_pair(const uint16_t* __restrict__ ga,
                                                         const uint16_t* __restrict__ gb,
                                                         float* __restrict__ acc, int64_t n_vec) {
    for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < n_vec;
         k += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = k * kVec;
        float xa[8], xb[8];
        widen8(ld_grad_u4(ga + i), xa);
        widen8(ld_grad_u4(gb + i), xb);
        F8 r;
        if (FIRST) {
#pragma unroll
            for (int j = 0; j < 8; ++j) r.v[j] = __fadd_rn(xa[j], xb[j]);
        } else {
            const F8 a = ld_state_f8(acc + i);
#pragma unroll
            for (int j = 0; j < 8; ++j) r.v[j] = __fadd_rn(__fadd_rn(a.v[j], xa[j]), xb[j]);
        }
        st_f8(acc + i, r);
    }
}

struct ViewArgs {
    void* views[DPG_MAX_VIEWS];
    int32_t n_views;
};

__global__ void __launch_bounds__(256) k_allgather(const float* __restrict__ master,
                                                   const __grid_constant__ ViewArgs va,
                                                   int64_t lo_vec, int64_t hi_vec) {
    for (int64_t k = lo_vec + int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < hi_vec;
         k += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = k * kVec;
        const F8 w = ld_grad_f8(master + i);
        const uint4 p = narrow8(w.v);
        for (int v = 0; v < va.n_views; ++v) st_u4(static_cast<uint16_t*>(va.views[v]) + i, p);
    }
}

// ZeRO-3 parameter all-gather: the bf16 shards (laid out in place in the flat
// parameter buffer) copied into every replica's full view; read once, written
// n_views times.
__global__ void __launch_bounds__(256) k_gather_bf16(const uint16_t* __restrict__ param,
                                                     const __grid_constant__ ViewArgs va,
                                                     int64_t lo_vec, int64_t hi_vec) {
    for (int64_t k = lo_vec + int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < hi_vec;
         k += int64_t(gridDim.x) * blockDim.x) {
        const uint4 x = ld_grad_u4(param + k * kVec);
        for (int v = 0; v < va.n_views; ++v) st_u4(static_cast<uint16_t*>(va.views[v]) + k * kVec, x);
    }
}

// ---------------------------------------------------------------------------
// pack / unpack: one CTA per item (<= kPackChunk elements of one parameter)
// ---------------------------------------------------------------------------
struct PackArgs {
    const void* ptrs[kPackPtrs];  // parameter gradients p_base .. p_base + kPackPtrs - 1
    int32_t p_base;
    int32_t unpack;
    const PackItem* items;
    int64_t item0;
    int64_t n_items;
    uint16_t* flat;
};

// Copy n bf16 elements.  When both ends are 16-byte aligned, each thread
// issues four 16-byte loads before its four stores, so a CTA keeps 64 KB in
// flight; otherwise (a parameter gradient at an odd 2-byte offset) it copies
// element by element.
__device__ __forceinline__ void copy_elems(uint16_t* __restrict__ dst,
                                           const uint16_t* __restrict__ src, int64_t n) {
    const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15) == 0;
    int64_t done = 0;
    if (vec) {
        const int64_t nv = n / kVec;
        const int64_t bd = blockDim.x;
        uint4* d4 = reinterpret_cast<uint4*>(dst);
        int64_t k = threadIdx.x;
        for (; k + 3 * bd < nv; k += 4 * bd) {
            const uint4 x0 = ld_grad_u4(src + (k) * kVec);
            const uint4 x1 = ld_grad_u4(src + (k + bd) * kVec);
            const uint4 x2 = ld_grad_u4(src + (k + 2 * bd) * kVec);
            const uint4 x3 = ld_grad_u4(src + (k + 3 * bd) * kVec);
            st_u4(d4 + k, x0);
            st_u4(d4 + k + bd, x1);
            st_u4(d4 + k + 2 * bd, x2);
            st_u4(d4 + k + 3 * bd, x3);
        }
        for (; k < nv; k += bd) st_u4(d4 + k, ld_grad_u4(src + k * kVec));
        done = nv * kVec;
    }
    for (int64_t k = done + threadIdx.x; k < n; k += blockDim.x) dst[k] = src[k];
}

// Persistent: CTA c copies items c, c + grid, ... of the launch's window.
__global__ void __launch_bounds__(256) k_pack(const __grid_constant__ PackArgs a) {
    for (int64_t j = blockIdx.x; j < a.n_items; j += gridDim.x) {
        const PackItem it = a.items[a.item0 + j];
        uint16_t* param = static_cast<uint16_t*>(const_cast<void*>(a.ptrs[it.param - a.p_base]));
        uint16_t* flat = a.flat + it.flat_off;
        if (!a.unpack) {
            if (it.count > 0) copy_elems(flat, param + it.src_off, it.count);
            for (int64_t k = threadIdx.x; k < it.tail; k += blockDim.x) flat[it.count + k] = 0;
        } else if (it.count > 0) {
            copy_elems(param + it.src_off, flat, it.count);
        }
    }
}

// ---------------------------------------------------------------------------
// checkpoint: fp32 state between the flat bucket layout and the canonical
// registration-order layout, one CTA per item (persistent)
// ---------------------------------------------------------------------------
struct StateArgs {
    const float* src[DPG_MAX_STATE_ARRAYS];
    float* dst[DPG_MAX_STATE_ARRAYS];
    int32_t n_arrays;
    int32_t to_flat;  // 1: canonical -> flat (import), 0: flat -> canonical
    const PackItem* items;
    int64_t n_items;
};

__device__ __forceinline__ void copy_f32(float* __restrict__ dst, const float* __restrict__ src,
                                         int64_t n) {
    const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15) == 0;
    int64_t done = 0;
    if (vec) {
        const int64_t n4 = n / 4;
        const float4* s4 = reinterpret_cast<const float4*>(src);
        float4* d4 = reinterpret_cast<float4*>(dst);
        for (int64_t k = threadIdx.x; k < n4; k += blockDim.x) d4[k] = __ldg(s4 + k);
        done = n4 * 4;
    }
    for (int64_t k = done + threadIdx.x; k < n; k += blockDim.x) dst[k] = __ldg(src + k);
}

__global__ void __launch_bounds__(256) k_state_copy(const __grid_constant__ StateArgs a) {
    for (int64_t j = blockIdx.x; j < a.n_items; j += gridDim.x) {
        const PackItem it = a.items[j];
        for (int k = 0; k < a.n_arrays; ++k) {
            if (a.to_flat) {
                float* flat = a.dst[k] + it.flat_off;
                if (it.count > 0) copy_f32(flat, a.src[k] + it.canon_off, it.count);
                for (int64_t e = threadIdx.x; e < it.tail; e += blockDim.x) flat[it.count + e] = 0.0f;
            } else if (it.count > 0) {
                copy_f32(a.dst[k] + it.canon_off, a.src[k] + it.flat_off, it.count);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------
static int sm_count(int dev, int* out) {
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
static int grid_cover(int64_t work_ctas, int* grid, const char* who) {
    if (work_ctas > 0x7FFFFFFF)
        return fail(DPG_ERR_INVALID_ARG, "%s: %lld CTAs in one launch", who, (long long)work_ctas);
    *grid = int(work_ctas > 0 ? work_ctas : 1);
    return DPG_OK;
}

// persistent-grid size: SM count x resident CTAs of `fn` (cached per device)
static int grid_for(const void* fn, int threads, int dev, int64_t work_ctas, int* grid) {
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

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

static int after_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(DPG_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return DPG_OK;
}

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Byte layout of a norm scratch with `visits` (CTA, bucket visit) slots for up
// to `ctas` CTAs; every section starts on a 256-byte boundary.
struct VisLayout {
    size_t sq, nf, bucket, count, total;
};

static VisLayout vis_layout(int64_t visits, int64_t ctas) {
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
    // chunked launches: tile -> bucket map, then the per-chunk norm partials
    const size_t n_tiles1 = size_t(p.n_tiles > 0 ? p.n_tiles : 1);
    const size_t n_chunks1 = n_tiles1 * kChunksPerTile;
    const size_t tb_bytes = round256(n_tiles1 * sizeof(int32_t));
    const size_t csq_bytes = round256(n_chunks1 * sizeof(double));
    void* chunk = nullptr;
    if (e == cudaSuccess) e = cudaMalloc(&chunk, tb_bytes + csq_bytes + n_chunks1 * sizeof(int32_t));
    std::vector<int32_t> tile_bucket(n_tiles1, 0);
    for (int32_t b = 0; b < p.n_buckets; ++b)
        for (int64_t t = p.tile_begin[b]; t < p.tile_begin[b + 1]; ++t) tile_bucket[size_t(t)] = b;
    if (e == cudaSuccess)
        e = cudaMemcpy(chunk, tile_bucket.data(), n_tiles1 * sizeof(int32_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(bo, p.bucket_offset.data(), nb1 * sizeof(int64_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(tb, p.tile_begin.data(), nb1 * sizeof(int64_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !p.items.empty())
        e = cudaMemcpy(it, p.items.data(), p.items.size() * sizeof(PackItem), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaFree(bo); cudaFree(tb); cudaFree(it); cudaFree(vis); cudaFree(clip); cudaFree(chunk);
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
    p.d_chunk = chunk;
    p.d_tile_bucket = static_cast<int32_t*>(chunk);
    p.d_chunk_sq = reinterpret_cast<double*>(static_cast<unsigned char*>(chunk) + tb_bytes);
    p.d_chunk_nf = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(chunk) + tb_bytes + csq_bytes);
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
    }
    if (have_cur) cudaSetDevice(cur);
    cudaGetLastError();
    p.device = -1;
}

// fp32 Adam constants, each computed in double and rounded once
static int adam_constants(const dpg_hparams* hp, RsAdamArgs& a) {
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
static int token_scale(const int64_t* tokens, int32_t n, float* scale) {
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

using RsKernel = void (*)(RsAdamArgs);

template <int MODE, int PHASE = kFull>
static RsKernel pick_rs_kernel(int R) {
    switch (R) {
        case 1: return k_rs_adam<1, MODE, PHASE>;
        case 2: return k_rs_adam<2, MODE, PHASE>;
        case 4: return k_rs_adam<4, MODE, PHASE>;
        case 8: return k_rs_adam<8, MODE, PHASE>;
        default: return k_rs_adam<0, MODE, PHASE>;
    }
}

template <int MODE>
static RsKernel pick_norm_kernel_r(int R) {
    switch (R) {
        case 1: return k_norm_pass<1, MODE>;
        case 2: return k_norm_pass<2, MODE>;
        case 4: return k_norm_pass<4, MODE>;
        case 8: return k_norm_pass<8, MODE>;
        default: return k_norm_pass<0, MODE>;
    }
}

static RsKernel pick_norm_kernel(int mode, int R) {
    return mode == kInBf16 ? pick_norm_kernel_r<kInBf16>(R)
         : mode == kInF32  ? pick_norm_kernel_r<kInF32>(R)
                           : pick_norm_kernel_r<kInF32PlusBf16>(R);
}

template <int PHASE>
static RsKernel pick_rs_kernel_mode(int mode, int R) {
    return mode == kInBf16 ? pick_rs_kernel<kInBf16, PHASE>(R)
         : mode == kInF32  ? pick_rs_kernel<kInF32, PHASE>(R)
                           : pick_rs_kernel<kInF32PlusBf16, PHASE>(R);
}

// Grid of a fused launch over tiles [t0, t1) and the visit slots per CTA it
// needs (a CTA visits at most every bucket of the range and at most one
// bucket per tile it processes).
static int fused_geometry(RsKernel fn, int dev, int64_t t0, int64_t t1, int32_t b0, int32_t b1,
                          int* grid, int32_t* vmax) {
    *grid = 0;
    *vmax = 0;
    if (t1 <= t0) return DPG_OK;
    int st = grid_for(reinterpret_cast<const void*>(fn), kThreads, dev, t1 - t0, grid);
    if (st != DPG_OK) return st;
    if (t_fused_max_ctas > 0 && *grid > t_fused_max_ctas) *grid = t_fused_max_ctas;
    const int64_t per_cta = (t1 - t0 + *grid - 1) / *grid;
    const int64_t buckets = int64_t(b1) - b0;
    *vmax = int32_t(per_cta < buckets ? per_cta : buckets);
    return DPG_OK;
}

// Launch the fused pass described by `a` (tables and, when a norm output is
// requested, norm scratch already filled in) on `grid` CTAs, then the norm
// finalize of buckets [a.b0, a.b1).
static int launch_fused(RsKernel fn, const RsAdamArgs& a, int grid, float* sqnorm,
                        int64_t* nonfinite, cudaStream_t s, const char* who,
                        double* sqnorm64 = nullptr) {
    int st = DPG_OK;
    if (a.t1 > a.t0) {
        cudaEvent_t ev0 = t_fused_start, ev1 = t_fused_stop;
        t_fused_start = t_fused_stop = nullptr;
        if (ev0) DPG_CUDA_TRY(cudaEventRecord(ev0, s));
        fn<<<grid, kThreads, 0, s>>>(a);
        st = after_launch(who);
        if (st != DPG_OK) return st;
        if (ev1) DPG_CUDA_TRY(cudaEventRecord(ev1, s));
    }
    if (sqnorm || nonfinite || sqnorm64) {
        const int32_t n_cta = a.t1 > a.t0 ? grid : 0;
        k_norm_finalize<<<a.b1 - a.b0, kFinalizeThreads, 0, s>>>(
            a.vis_sq, a.vis_nf, a.vis_bucket, a.vis_count, n_cta, a.vmax, a.b0, sqnorm, nonfinite,
            sqnorm64);
        st = after_launch(who);
    }
    return st;
}

template <int MODE, int PHASE = kFull>
static RsKernel pick_chunk_kernel(int R) {
    switch (R) {
        case 1: return k_rs_adam_chunk<1, MODE, PHASE>;
        case 2: return k_rs_adam_chunk<2, MODE, PHASE>;
        case 4: return k_rs_adam_chunk<4, MODE, PHASE>;
        case 8: return k_rs_adam_chunk<8, MODE, PHASE>;
        default: return k_rs_adam_chunk<0, MODE, PHASE>;
    }
}

// CTA size of the chunked norm pass (128, 256 and 512 threads measured; the
// smallest is fastest, as for the fused pass).
constexpr int kNormChunkThreads = 128;

template <int MODE>
static RsKernel pick_norm_chunk_kernel(int R) {
    switch (R) {
        case 1: return k_norm_chunk<1, MODE, kNormChunkThreads>;
        case 2: return k_norm_chunk<2, MODE, kNormChunkThreads>;
        case 4: return k_norm_chunk<4, MODE, kNormChunkThreads>;
        case 8: return k_norm_chunk<8, MODE, kNormChunkThreads>;
        default: return k_norm_chunk<0, MODE, kNormChunkThreads>;
    }
}

// Chunked launch of the fused pass over tiles [a.t0, a.t1) (tables already in
// `a`), then, when a norm output is requested, the per-bucket finalize.
static int launch_chunked(RsKernel fn, RsAdamArgs a, const Plan& p, bool want_norm, float* sqnorm,
                          int64_t* nonfinite, cudaStream_t s, const char* who,
                          double* sqnorm64 = nullptr, int threads = kChunkThreads) {
    const int cpt = int(kTile / (int64_t(threads) * kVec));   // chunks per tile
    a.tile_bucket = p.d_tile_bucket;
    a.chunk_sq = want_norm ? p.d_chunk_sq : nullptr;
    a.chunk_nf = want_norm ? p.d_chunk_nf : nullptr;
    const int64_t n_chunks = (a.t1 - a.t0) * cpt;
    if (n_chunks > 0x7FFFFFFF) return fail(DPG_ERR_INVALID_ARG, "%s: %lld chunks in one launch", who,
                                           (long long)n_chunks);
    int st = DPG_OK;
    if (n_chunks > 0) {
        cudaEvent_t ev0 = t_fused_start, ev1 = t_fused_stop;
        t_fused_start = t_fused_stop = nullptr;
        if (ev0) DPG_CUDA_TRY(cudaEventRecord(ev0, s));
        fn<<<unsigned(n_chunks), threads, 0, s>>>(a);
        st = after_launch(who);
        if (st != DPG_OK) return st;
        if (ev1) DPG_CUDA_TRY(cudaEventRecord(ev1, s));
    }
    if (want_norm) {
        k_chunk_finalize<<<a.b1 - a.b0, kChunkFinalizeThreads, 0, s>>>(
            p.d_chunk_sq, p.d_chunk_nf, p.d_tile_begin, a.t0, cpt, a.b0, sqnorm, nonfinite, sqnorm64);
        st = after_launch(who);
    }
    return st;
}

static int rs_adam(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                   const void* const* last, const int64_t* tokens, int32_t n_counts,
                   const dpg_hparams* hp, float* master, float* m, float* v,
                   void* const* views, int32_t n_views, float* sqnorm, int64_t* nonfinite,
                   float* reduced, int32_t b0, int32_t b1, void* stream, const char* who,
                   const void* const* last2 = nullptr) {
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "%s: plan is NULL", who);
    Plan& p = const_cast<dpg_plan_t*>(plan)->p;
    if (b0 < 0 || b1 < b0 || b1 > p.n_buckets)
        return fail(DPG_ERR_INVALID_ARG, "%s: bucket range [%d, %d) outside [0, %d]", who, b0, b1,
                    p.n_buckets);
    if (grads_dtype != DPG_BF16 && grads_dtype != DPG_F32)
        return fail(DPG_ERR_INVALID_ARG, "%s: grads_dtype %d unknown", who, grads_dtype);
    if (last && grads_dtype != DPG_F32)
        return fail(DPG_ERR_INVALID_ARG, "%s: last_micro_bf16 needs fp32 accumulation grads", who);
    if (last2 && !last)
        return fail(DPG_ERR_INVALID_ARG, "%s: the final microbatch needs the one before it", who);
    if (n_views < 0 || n_views > DPG_MAX_VIEWS)
        return fail(DPG_ERR_INVALID_ARG, "%s: n_views %d outside [0, %d]", who, n_views, DPG_MAX_VIEWS);
    RsAdamArgs a{};
    int st = adam_constants(hp, a);
    if (st != DPG_OK) return st;
    st = token_scale(tokens, n_counts, &a.scale);
    if (st != DPG_OK) return st;
    if (b0 == b1) return DPG_OK;  // nothing to update; buffers are not touched
    const bool want_norm = sqnorm || nonfinite;
    const bool has_elems = p.bucket_offset[b1] > p.bucket_offset[b0];
    if (!has_elems && !want_norm) return DPG_OK;
    if (!has_elems) n_views = 0;  // only the (zero) norms of empty buckets are written
    if (has_elems && !grads) return fail(DPG_ERR_INVALID_ARG, "%s: grads is NULL", who);
    if (has_elems && (!master || !m || !v))
        return fail(DPG_ERR_INVALID_ARG, "%s: master/m/v must not be NULL", who);
    if (n_views > 0 && !views) return fail(DPG_ERR_INVALID_ARG, "%s: param_views is NULL", who);
    const uintptr_t galign = grads_dtype == DPG_BF16 ? 16 : 32;
    for (int r = 0; has_elems && r < p.R; ++r) {
        if (!grads[r]) return fail(DPG_ERR_INVALID_ARG, "%s: grads[%d] is NULL", who, r);
        if (!aligned(grads[r], galign)) return fail(DPG_ERR_MISALIGNED, "%s: grads[%d] misaligned", who, r);
        a.grads[r] = grads[r];
        if (last) {
            if (!last[r]) return fail(DPG_ERR_INVALID_ARG, "%s: last_micro_bf16[%d] is NULL", who, r);
            if (!aligned(last[r], 16)) return fail(DPG_ERR_MISALIGNED, "%s: last_micro_bf16[%d] misaligned", who, r);
            a.last[r] = last[r];
        }
        if (last2) {
            if (!last2[r]) return fail(DPG_ERR_INVALID_ARG, "%s: final microbatch[%d] is NULL", who, r);
            if (!aligned(last2[r], 16)) return fail(DPG_ERR_MISALIGNED, "%s: final microbatch[%d] misaligned", who, r);
            a.last2[r] = last2[r];
        }
    }
    for (int k = 0; k < n_views; ++k) {
        if (!views[k]) return fail(DPG_ERR_INVALID_ARG, "%s: param_views[%d] is NULL", who, k);
        if (!aligned(views[k], 16)) return fail(DPG_ERR_MISALIGNED, "%s: param_views[%d] misaligned", who, k);
        a.views[k] = views[k];
    }
    if (!aligned(master, 32) || !aligned(m, 32) || !aligned(v, 32) || !aligned(reduced, 32))
        return fail(DPG_ERR_MISALIGNED, "%s: fp32 buffers must be 32-byte aligned", who);
    st = upload(p);
    if (st != DPG_OK) return st;

    a.master = master;
    a.m = m;
    a.v = v;
    a.reduced = reduced;
    a.bucket_offset = p.d_bucket_offset;
    a.tile_begin = p.d_tile_begin;
    a.t0 = p.tile_begin[b0];
    a.t1 = p.tile_begin[b1];
    a.b0 = b0;
    a.b1 = b1;
    a.R = p.R;
    a.n_views = n_views;
    const int mode = grads_dtype == DPG_BF16 ? kInBf16
                   : last2 ? kInF32PlusBf16x2 : (last ? kInF32PlusBf16 : kInF32);
    if (t_fused_max_ctas == 0) {
        RsKernel fc = mode == kInBf16 ? pick_chunk_kernel<kInBf16>(p.R)
                    : mode == kInF32 ? pick_chunk_kernel<kInF32>(p.R)
                    : mode == kInF32PlusBf16 ? pick_chunk_kernel<kInF32PlusBf16>(p.R)
                                             : pick_chunk_kernel<kInF32PlusBf16x2>(p.R);
        return launch_chunked(fc, a, p, want_norm, sqnorm, nonfinite,
                              static_cast<cudaStream_t>(stream), who);
    }
    // a grid cap asks for the persistent kernel, whose CTA count it bounds
    RsKernel fn = mode == kInBf16 ? pick_rs_kernel<kInBf16>(p.R)
                : mode == kInF32 ? pick_rs_kernel<kInF32>(p.R)
                : mode == kInF32PlusBf16 ? pick_rs_kernel<kInF32PlusBf16>(p.R)
                                         : pick_rs_kernel<kInF32PlusBf16x2>(p.R);
    int grid = 0;
    st = fused_geometry(fn, p.device, a.t0, a.t1, b0, b1, &grid, &a.vmax);
    if (st != DPG_OK) return st;
    if (want_norm) {
        if (grid > p.cap_ctas || int64_t(grid) * a.vmax > p.cap_visits)
            return fail(DPG_ERR_CUDA, "%s: norm scratch too small (%d CTAs x %d visits)", who,
                        grid, a.vmax);
        a.vis_sq = p.d_vis_sq;
        a.vis_nf = p.d_vis_nf;
        a.vis_bucket = p.d_vis_bucket;
        a.vis_count = p.d_vis_count;
    }
    return launch_fused(fn, a, grid, sqnorm, nonfinite, static_cast<cudaStream_t>(stream), who);
}

// Validate the per-call buffers of a whole-plan step and copy them into `a`.
static int fill_step_args(const Plan& p, const void* const* grads, int32_t grads_dtype,
                          const void* const* last, const dpg_hparams* hp, const int64_t* tokens,
                          int32_t n_counts, float* master, float* m, float* v,
                          void* const* views, int32_t n_views, RsAdamArgs& a, const char* who) {
    if (grads_dtype != DPG_BF16 && grads_dtype != DPG_F32)
        return fail(DPG_ERR_INVALID_ARG, "%s: grads_dtype %d unknown", who, grads_dtype);
    if (last && grads_dtype != DPG_F32)
        return fail(DPG_ERR_INVALID_ARG, "%s: last_micro_bf16 needs fp32 accumulation grads", who);
    if (n_views < 0 || n_views > DPG_MAX_VIEWS)
        return fail(DPG_ERR_INVALID_ARG, "%s: n_views %d outside [0, %d]", who, n_views, DPG_MAX_VIEWS);
    int st = adam_constants(hp, a);
    if (st != DPG_OK) return st;
    st = token_scale(tokens, n_counts, &a.scale);
    if (st != DPG_OK) return st;
    const bool has_elems = p.total_padded > 0;
    if (!has_elems) n_views = 0;
    if (has_elems && !grads) return fail(DPG_ERR_INVALID_ARG, "%s: grads is NULL", who);
    if (has_elems && (!master || !m || !v))
        return fail(DPG_ERR_INVALID_ARG, "%s: master/m/v must not be NULL", who);
    if (n_views > 0 && !views) return fail(DPG_ERR_INVALID_ARG, "%s: param_views is NULL", who);
    const uintptr_t galign = grads_dtype == DPG_BF16 ? 16 : 32;
    for (int r = 0; has_elems && r < p.R; ++r) {
        if (!grads[r]) return fail(DPG_ERR_INVALID_ARG, "%s: grads[%d] is NULL", who, r);
        if (!aligned(grads[r], galign)) return fail(DPG_ERR_MISALIGNED, "%s: grads[%d] misaligned", who, r);
        a.grads[r] = grads[r];
        if (last) {
            if (!last[r]) return fail(DPG_ERR_INVALID_ARG, "%s: last_micro_bf16[%d] is NULL", who, r);
            if (!aligned(last[r], 16)) return fail(DPG_ERR_MISALIGNED, "%s: last_micro_bf16[%d] misaligned", who, r);
            a.last[r] = last[r];
        }
    }
    for (int k = 0; k < n_views; ++k) {
        if (!views[k]) return fail(DPG_ERR_INVALID_ARG, "%s: param_views[%d] is NULL", who, k);
        if (!aligned(views[k], 16)) return fail(DPG_ERR_MISALIGNED, "%s: param_views[%d] misaligned", who, k);
        a.views[k] = views[k];
    }
    if (!aligned(master, 32) || !aligned(m, 32) || !aligned(v, 32))
        return fail(DPG_ERR_MISALIGNED, "%s: fp32 buffers must be 32-byte aligned", who);
    a.master = master;
    a.m = m;
    a.v = v;
    a.n_views = n_views;
    a.R = p.R;
    return DPG_OK;
}

// Whole step with global gradient-norm clipping: norm pass, coefficient on
// the device, update pass (see dpg_step_clipped in include/dpg.h).
static int step_clipped(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                        const void* const* last, const int64_t* tokens, int32_t n_counts,
                        const dpg_hparams* hp, double max_norm, float* master, float* m,
                        float* v, void* const* views, int32_t n_views, float* sqnorm,
                        int64_t* nonfinite, float* reduced, float* clip_out, void* stream) {
    const char* who = "dpg_step_clipped";
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "%s: plan is NULL", who);
    Plan& p = const_cast<dpg_plan_t*>(plan)->p;
    if (!(max_norm > 0.0) || !std::isfinite(max_norm))
        return fail(DPG_ERR_INVALID_ARG, "%s: max_norm must be finite and > 0", who);
    RsAdamArgs a{};
    int st = fill_step_args(p, grads, grads_dtype, last, hp, tokens, n_counts, master, m, v, views,
                            n_views, a, who);
    if (st != DPG_OK) return st;
    if (!aligned(reduced, 32)) return fail(DPG_ERR_MISALIGNED, "%s: reduced_grad misaligned", who);
    if (p.n_buckets == 0) return DPG_OK;
    st = upload(p);
    if (st != DPG_OK) return st;
    a.bucket_offset = p.d_bucket_offset;
    a.tile_begin = p.d_tile_begin;
    a.t0 = 0;
    a.t1 = p.n_tiles;
    a.b0 = 0;
    a.b1 = p.n_buckets;
    const int mode = grads_dtype == DPG_BF16 ? kInBf16 : (last ? kInF32PlusBf16 : kInF32);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // pass 1: reduce, scale, exact squares per bucket (and g, when a buffer is given)
    RsAdamArgs a1 = a;
    a1.reduced = reduced;
    // Chunked unless a grid cap is set -- or when the pass only reads the
    // replicas (no g stored) and R <= 4: then it moves just 2R bytes per
    // element, and the persistent pass, which keeps up to four tiles' loads
    // in flight per thread, is faster (4.5B, R = 4: 27.3 against 28.5 ms
    // for the whole step).
    if (t_fused_max_ctas == 0 && (reduced != nullptr || p.R >= 8)) {
        RsKernel fc1 = mode == kInBf16 ? pick_norm_chunk_kernel<kInBf16>(p.R)
                     : mode == kInF32  ? pick_norm_chunk_kernel<kInF32>(p.R)
                                       : pick_norm_chunk_kernel<kInF32PlusBf16>(p.R);
        st = launch_chunked(fc1, a1, p, true, sqnorm, nonfinite, s, who, p.d_bucket_sq64,
                            kNormChunkThreads);
    } else {   // the persistent norm pass
        RsKernel fn1 = pick_norm_kernel(mode, p.R);
        int grid1 = 0;
        st = fused_geometry(fn1, p.device, a1.t0, a1.t1, 0, p.n_buckets, &grid1, &a1.vmax);
        if (st != DPG_OK) return st;
        if (grid1 > p.cap_ctas || int64_t(grid1) * a1.vmax > p.cap_visits)
            return fail(DPG_ERR_CUDA, "%s: norm scratch too small", who);
        a1.vis_sq = p.d_vis_sq;
        a1.vis_nf = p.d_vis_nf;
        a1.vis_bucket = p.d_vis_bucket;
        a1.vis_count = p.d_vis_count;
        if (a1.t1 > a1.t0) {
            fn1<<<grid1, kThreads, 0, s>>>(a1);
            st = after_launch(who);
            if (st != DPG_OK) return st;
        }
        k_norm_finalize<<<p.n_buckets, kFinalizeThreads, 0, s>>>(
            a1.vis_sq, a1.vis_nf, a1.vis_bucket, a1.vis_count, a1.t1 > a1.t0 ? grid1 : 0, a1.vmax, 0,
            sqnorm, nonfinite, p.d_bucket_sq64);
        st = after_launch(who);
    }
    if (st != DPG_OK) return st;
    // the coefficient, on the device: no host synchronisation
    k_clip_coef<<<1, 256, 0, s>>>(p.d_bucket_sq64, p.n_buckets, max_norm, p.d_clip_coef, clip_out);
    st = after_launch(who);
    if (st != DPG_OK) return st;
    // pass 2: g * coef -> Adam -> bf16 views, from the stored g or the replicas again
    RsAdamArgs a2 = a;
    a2.clip_coef = p.d_clip_coef;
    if (t_fused_max_ctas == 0) {
        RsKernel fc;
        if (reduced) {
            a2.g_in = reduced;
            fc = k_rs_adam_chunk<1, kInReduced, kUpdate>;
        } else {
            fc = mode == kInBf16 ? pick_chunk_kernel<kInBf16, kUpdate>(p.R)
               : mode == kInF32  ? pick_chunk_kernel<kInF32, kUpdate>(p.R)
                                 : pick_chunk_kernel<kInF32PlusBf16, kUpdate>(p.R);
        }
        return launch_chunked(fc, a2, p, false, nullptr, nullptr, s, who);
    }
    RsKernel fn2;
    if (reduced) {
        a2.g_in = reduced;
        fn2 = k_rs_adam<1, kInReduced, kUpdate>;
    } else {
        fn2 = pick_rs_kernel_mode<kUpdate>(mode, p.R);
    }
    int grid2 = 0;
    st = fused_geometry(fn2, p.device, a2.t0, a2.t1, 0, p.n_buckets, &grid2, &a2.vmax);
    if (st != DPG_OK) return st;
    return launch_fused(fn2, a2, grid2, nullptr, nullptr, s, who);
}

// All-reduce of the replica gradients (DDP): every element's rank-ordered
// sum times fp32(1/G), written to `reduced`; optional per-bucket norms.
static int allreduce_grads(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                           const void* const* last, const int64_t* tokens, int32_t n_counts,
                           float* reduced, float* sqnorm, int64_t* nonfinite, int32_t b0,
                           int32_t b1, void* stream) {
    const char* who = "dpg_allreduce_grads";
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "%s: plan is NULL", who);
    Plan& p = const_cast<dpg_plan_t*>(plan)->p;
    if (b0 < 0 || b1 < b0 || b1 > p.n_buckets)
        return fail(DPG_ERR_INVALID_ARG, "%s: bucket range [%d, %d) outside [0, %d]", who, b0, b1,
                    p.n_buckets);
    if (grads_dtype != DPG_BF16 && grads_dtype != DPG_F32)
        return fail(DPG_ERR_INVALID_ARG, "%s: grads_dtype %d unknown", who, grads_dtype);
    if (last && grads_dtype != DPG_F32)
        return fail(DPG_ERR_INVALID_ARG, "%s: last_micro_bf16 needs fp32 accumulation grads", who);
    RsAdamArgs a{};
    int st = token_scale(tokens, n_counts, &a.scale);
    if (st != DPG_OK) return st;
    if (b0 == b1) return DPG_OK;
    const bool want_norm = sqnorm || nonfinite;
    const bool has_elems = p.bucket_offset[b1] > p.bucket_offset[b0];
    if (!has_elems && !want_norm) return DPG_OK;
    if (has_elems) {
        if (!grads) return fail(DPG_ERR_INVALID_ARG, "%s: grads is NULL", who);
        if (!reduced) return fail(DPG_ERR_INVALID_ARG, "%s: reduced_grad is NULL", who);
        if (!aligned(reduced, 32)) return fail(DPG_ERR_MISALIGNED, "%s: reduced_grad misaligned", who);
        const uintptr_t galign = grads_dtype == DPG_BF16 ? 16 : 32;
        for (int r = 0; r < p.R; ++r) {
            if (!grads[r]) return fail(DPG_ERR_INVALID_ARG, "%s: grads[%d] is NULL", who, r);
            if (!aligned(grads[r], galign)) return fail(DPG_ERR_MISALIGNED, "%s: grads[%d] misaligned", who, r);
            a.grads[r] = grads[r];
            if (last) {
                if (!last[r]) return fail(DPG_ERR_INVALID_ARG, "%s: last_micro_bf16[%d] is NULL", who, r);
                if (!aligned(last[r], 16)) return fail(DPG_ERR_MISALIGNED, "%s: last_micro_bf16[%d] misaligned", who, r);
                a.last[r] = last[r];
            }
        }
    }
    st = upload(p);
    if (st != DPG_OK) return st;
    a.reduced = reduced;
    a.bucket_offset = p.d_bucket_offset;
    a.tile_begin = p.d_tile_begin;
    a.t0 = p.tile_begin[b0];
    a.t1 = p.tile_begin[b1];
    a.b0 = b0;
    a.b1 = b1;
    a.R = p.R;
    const int mode = grads_dtype == DPG_BF16 ? kInBf16 : (last ? kInF32PlusBf16 : kInF32);
    if (t_fused_max_ctas == 0 && has_elems) {
        RsKernel fc = mode == kInBf16 ? pick_chunk_kernel<kInBf16, kNormOnly>(p.R)
                    : mode == kInF32  ? pick_chunk_kernel<kInF32, kNormOnly>(p.R)
                                      : pick_chunk_kernel<kInF32PlusBf16, kNormOnly>(p.R);
        return launch_chunked(fc, a, p, want_norm, sqnorm, nonfinite,
                              static_cast<cudaStream_t>(stream), who);
    }
    RsKernel fn = pick_norm_kernel(mode, p.R);
    int grid = 0;
    st = fused_geometry(fn, p.device, a.t0, a.t1, b0, b1, &grid, &a.vmax);
    if (st != DPG_OK) return st;
    if (want_norm) {
        if (grid > p.cap_ctas || int64_t(grid) * a.vmax > p.cap_visits)
            return fail(DPG_ERR_CUDA, "%s: norm scratch too small", who);
        a.vis_sq = p.d_vis_sq;
        a.vis_nf = p.d_vis_nf;
        a.vis_bucket = p.d_vis_bucket;
        a.vis_count = p.d_vis_count;
    }
    return launch_fused(fn, a, grid, sqnorm, nonfinite, static_cast<cudaStream_t>(stream), who);
}

// One replica's optimizer step from an already-reduced gradient (DDP /
// NO_SHARD: every replica updates its own full copy of the state).
static int adam_from_reduced(const dpg_plan_t* plan, const float* reduced, const dpg_hparams* hp,
                             float* master, float* m, float* v, void* const* views,
                             int32_t n_views, float* sqnorm, int64_t* nonfinite, int32_t b0,
                             int32_t b1, void* stream) {
    const char* who = "dpg_adam_from_reduced";
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "%s: plan is NULL", who);
    Plan& p = const_cast<dpg_plan_t*>(plan)->p;
    if (b0 < 0 || b1 < b0 || b1 > p.n_buckets)
        return fail(DPG_ERR_INVALID_ARG, "%s: bucket range [%d, %d) outside [0, %d]", who, b0, b1,
                    p.n_buckets);
    if (n_views < 0 || n_views > DPG_MAX_VIEWS)
        return fail(DPG_ERR_INVALID_ARG, "%s: n_views %d outside [0, %d]", who, n_views, DPG_MAX_VIEWS);
    RsAdamArgs a{};
    int st = adam_constants(hp, a);
    if (st != DPG_OK) return st;
    if (b0 == b1) return DPG_OK;
    const bool want_norm = sqnorm || nonfinite;
    const bool has_elems = p.bucket_offset[b1] > p.bucket_offset[b0];
    if (!has_elems && !want_norm) return DPG_OK;
    if (!has_elems) n_views = 0;
    if (has_elems) {
        if (!reduced || !master || !m || !v)
            return fail(DPG_ERR_INVALID_ARG, "%s: reduced_grad/master/m/v must not be NULL", who);
        if (!aligned(reduced, 32) || !aligned(master, 32) || !aligned(m, 32) || !aligned(v, 32))
            return fail(DPG_ERR_MISALIGNED, "%s: fp32 buffers must be 32-byte aligned", who);
    }
    if (n_views > 0 && !views) return fail(DPG_ERR_INVALID_ARG, "%s: param_views is NULL", who);
    for (int k = 0; k < n_views; ++k) {
        if (!views[k]) return fail(DPG_ERR_INVALID_ARG, "%s: param_views[%d] is NULL", who, k);
        if (!aligned(views[k], 16)) return fail(DPG_ERR_MISALIGNED, "%s: param_views[%d] misaligned", who, k);
        a.views[k] = views[k];
    }
    st = upload(p);
    if (st != DPG_OK) return st;
    a.g_in = reduced;
    a.master = master;
    a.m = m;
    a.v = v;
    a.n_views = n_views;
    a.bucket_offset = p.d_bucket_offset;
    a.tile_begin = p.d_tile_begin;
    a.t0 = p.tile_begin[b0];
    a.t1 = p.tile_begin[b1];
    a.b0 = b0;
    a.b1 = b1;
    a.R = p.R;
    if (t_fused_max_ctas == 0)
        return launch_chunked(k_rs_adam_chunk<1, kInReduced, kFull>, a, p, want_norm, sqnorm,
                              nonfinite, static_cast<cudaStream_t>(stream), who);
    RsKernel fn = k_rs_adam<1, kInReduced, kFull>;
    int grid = 0;
    st = fused_geometry(fn, p.device, a.t0, a.t1, b0, b1, &grid, &a.vmax);
    if (st != DPG_OK) return st;
    if (want_norm) {
        if (grid > p.cap_ctas || int64_t(grid) * a.vmax > p.cap_visits)
            return fail(DPG_ERR_CUDA, "%s: norm scratch too small", who);
        a.vis_sq = p.d_vis_sq;
        a.vis_nf = p.d_vis_nf;
        a.vis_bucket = p.d_vis_bucket;
        a.vis_count = p.d_vis_count;
    }
    return launch_fused(fn, a, grid, sqnorm, nonfinite, static_cast<cudaStream_t>(stream), who);
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
        k_norm_finalize<<<p.n_buckets, kFinalizeThreads, 0, s>>>(
            a.vis_sq, a.vis_nf, a.vis_bucket, a.vis_count, units > 0 ? grid : 0, a.vmax, 0, sqnorm,
            nonfinite, nullptr);
        st = after_launch(who);
    }
    return st;
}

}  // namespace dpg

using dpg::fail;

extern "C" {

int64_t dpg_launch_count(void) { return dpg::g_launches.load(); }

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

int dpg_allreduce_grads(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                        const void* const* last_micro_bf16, const int64_t* valid_tokens,
                        int32_t n_counts, float* reduced_grad, float* bucket_sqnorm,
                        int64_t* bucket_nonfinite, int32_t b0, int32_t b1, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_allreduce_grads");
    return dpg::allreduce_grads(plan, grads, grads_dtype, last_micro_bf16, valid_tokens, n_counts,
                                reduced_grad, bucket_sqnorm, bucket_nonfinite, b0, b1, stream);
}

int dpg_adam_from_reduced(const dpg_plan_t* plan, const float* reduced_grad, const dpg_hparams* hp,
                          float* master, float* exp_avg, float* exp_avg_sq,
                          void* const* param_views, int32_t n_views, float* bucket_sqnorm,
                          int64_t* bucket_nonfinite, int32_t b0, int32_t b1, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_adam_from_reduced");
    return dpg::adam_from_reduced(plan, reduced_grad, hp, master, exp_avg, exp_avg_sq, param_views,
                                  n_views, bucket_sqnorm, bucket_nonfinite, b0, b1, stream);
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
    dpg::t_staged_skip = skip_unit;
    dpg::t_staged_timeout_ns = timeout_ns;
    return DPG_OK;
}

int dpg_step_clipped(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                     const void* const* last_micro_bf16, const int64_t* valid_tokens,
                     int32_t n_counts, const dpg_hparams* hp, double max_norm, float* master,
                     float* exp_avg, float* exp_avg_sq, void* const* param_views, int32_t n_views,
                     float* bucket_sqnorm, int64_t* bucket_nonfinite, float* reduced_grad,
                     float* clip_out, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_step_clipped");
    return dpg::step_clipped(plan, grads, grads_dtype, last_micro_bf16, valid_tokens, n_counts, hp,
                             max_norm, master, exp_avg, exp_avg_sq, param_views, n_views,
                             bucket_sqnorm, bucket_nonfinite, reduced_grad, clip_out, stream);
}

int dpg_set_fused_max_ctas(int32_t max_ctas) {
    dpg::clear_error();
    if (max_ctas < 0) return fail(DPG_ERR_INVALID_ARG, "dpg_set_fused_max_ctas: %d < 0", max_ctas);
    dpg::t_fused_max_ctas = max_ctas;
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

int dpg_reduce_scatter_adam(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                            const void* const* last_micro_bf16, const int64_t* valid_tokens,
                            int32_t n_counts, const dpg_hparams* hp, float* master,
                            float* exp_avg, float* exp_avg_sq, void* const* param_views,
                            int32_t n_views, float* bucket_sqnorm, int64_t* bucket_nonfinite,
                            float* reduced_grad, int32_t b0, int32_t b1, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_reduce_scatter_adam");
    return dpg::rs_adam(plan, grads, grads_dtype, last_micro_bf16, valid_tokens, n_counts, hp,
                        master, exp_avg, exp_avg_sq, param_views, n_views, bucket_sqnorm,
                        bucket_nonfinite, reduced_grad, b0, b1, stream, "dpg_reduce_scatter_adam");
}

int dpg_step(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
             const void* const* last_micro_bf16, const int64_t* valid_tokens, int32_t n_counts,
             const dpg_hparams* hp, float* master, float* exp_avg, float* exp_avg_sq,
             void* const* param_views, int32_t n_views, float* bucket_sqnorm,
             int64_t* bucket_nonfinite, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_step");
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_step: plan is NULL");
    return dpg::rs_adam(plan, grads, grads_dtype, last_micro_bf16, valid_tokens, n_counts, hp,
                        master, exp_avg, exp_avg_sq, param_views, n_views, bucket_sqnorm,
                        bucket_nonfinite, nullptr, 0, plan->p.n_buckets, stream, "dpg_step");
}

int dpg_accumulate(const dpg_plan_t* plan, const void* flat_bf16, float* acc_f32, int32_t first,
                   void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_accumulate");
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_accumulate: plan is NULL");
    if (plan->p.total_padded == 0) return DPG_OK;
    if (!flat_bf16 || !acc_f32) return fail(DPG_ERR_INVALID_ARG, "dpg_accumulate: NULL buffer");
    if (!dpg::aligned(flat_bf16, 16) || !dpg::aligned(acc_f32, 32))
        return fail(DPG_ERR_MISALIGNED, "dpg_accumulate: misaligned buffer");
    dpg::Plan& p = const_cast<dpg_plan_t*>(plan)->p;
    const int64_t n_vec = p.total_padded / dpg::kVec;
    if (n_vec == 0) return DPG_OK;
    int grid = 0;
    int st = dpg::grid_cover((n_vec + 255) / 256, &grid, "dpg_accumulate");
    if (st != DPG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint16_t* g = static_cast<const uint16_t*>(flat_bf16);
    if (first) dpg::k_accumulate<true><<<grid, 256, 0, s>>>(g, acc_f32, n_vec);
    else dpg::k_accumulate<false><<<grid, 256, 0, s>>>(g, acc_f32, n_vec);
    return dpg::after_launch("dpg_accumulate");
}

int dpg_accumulate_pair(const dpg_plan_t* plan, const void* micro_a_bf16, const void* micro_b_bf16,
                        float* acc_f32, int32_t first, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_accumulate_pair");
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_accumulate_pair: plan is NULL");
    if (plan->p.total_padded == 0) return DPG_OK;
    if (!micro_a_bf16 || !micro_b_bf16 || !acc_f32)
        return fail(DPG_ERR_INVALID_ARG, "dpg_accumulate_pair: NULL buffer");
    if (!dpg::aligned(micro_a_bf16, 16) || !dpg::aligned(micro_b_bf16, 16) || !dpg::aligned(acc_f32, 32))
        return fail(DPG_ERR_MISALIGNED, "dpg_accumulate_pair: misaligned buffer");
    const dpg::Plan& p = plan->p;
    const int64_t n_vec = p.total_padded / dpg::kVec;
    int grid = 0;
    int st = dpg::grid_cover((n_vec + 255) / 256, &grid, "dpg_accumulate_pair");
    if (st != DPG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint16_t* ga = static_cast<const uint16_t*>(micro_a_bf16);
    const uint16_t* gb = static_cast<const uint16_t*>(micro_b_bf16);
    if (first) dpg::k_accumulate_pair<true><<<grid, 256, 0, s>>>(ga, gb, acc_f32, n_vec);
    else dpg::k_accumulate_pair<false><<<grid, 256, 0, s>>>(ga, gb, acc_f32, n_vec);
    return dpg::after_launch("dpg_accumulate_pair");
}

int dpg_step_fold2(const dpg_plan_t* plan, const float* const* acc_f32,
                   const void* const* micro_a_bf16, const void* const* micro_b_bf16,
                   const int64_t* valid_tokens, int32_t n_counts, const dpg_hparams* hp,
                   float* master, float* exp_avg, float* exp_avg_sq, void* const* param_views,
                   int32_t n_views, float* bucket_sqnorm, int64_t* bucket_nonfinite,
                   void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_step_fold2");
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_step_fold2: plan is NULL");
    if (!micro_a_bf16 || !micro_b_bf16)
        return fail(DPG_ERR_INVALID_ARG, "dpg_step_fold2: microbatch tables must not be NULL");
    return dpg::rs_adam(plan, reinterpret_cast<const void* const*>(acc_f32), DPG_F32, micro_a_bf16,
                        valid_tokens, n_counts, hp, master, exp_avg, exp_avg_sq, param_views,
                        n_views, bucket_sqnorm, bucket_nonfinite, nullptr, 0, plan->p.n_buckets,
                        stream, "dpg_step_fold2", micro_b_bf16);
}

int dpg_allgather_params(const dpg_plan_t* plan, const float* master, void* const* views,
                         int32_t n_views, int32_t b0, int32_t b1, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_allgather_params");
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_allgather_params: plan is NULL");
    const dpg::Plan& p = plan->p;
    if (b0 < 0 || b1 < b0 || b1 > p.n_buckets)
        return fail(DPG_ERR_INVALID_ARG, "dpg_allgather_params: bucket range [%d, %d) outside [0, %d]",
                    b0, b1, p.n_buckets);
    if (n_views < 0 || n_views > DPG_MAX_VIEWS)
        return fail(DPG_ERR_INVALID_ARG, "dpg_allgather_params: n_views %d outside [0, %d]", n_views,
                    DPG_MAX_VIEWS);
    if (b0 == b1 || n_views == 0 || p.bucket_offset[b1] == p.bucket_offset[b0]) return DPG_OK;
    if (!master) return fail(DPG_ERR_INVALID_ARG, "dpg_allgather_params: master is NULL");
    if (!dpg::aligned(master, 32)) return fail(DPG_ERR_MISALIGNED, "dpg_allgather_params: master misaligned");
    if (n_views > 0 && !views) return fail(DPG_ERR_INVALID_ARG, "dpg_allgather_params: views is NULL");
    dpg::ViewArgs va{};
    va.n_views = n_views;
    for (int k = 0; k < n_views; ++k) {
        if (!views[k]) return fail(DPG_ERR_INVALID_ARG, "dpg_allgather_params: views[%d] is NULL", k);
        if (!dpg::aligned(views[k], 16))
            return fail(DPG_ERR_MISALIGNED, "dpg_allgather_params: views[%d] misaligned", k);
        va.views[k] = views[k];
    }
    const int64_t lo = p.bucket_offset[b0] / dpg::kVec, hi = p.bucket_offset[b1] / dpg::kVec;
    if (hi <= lo || n_views == 0) return DPG_OK;
    int grid = 0;
    int st = dpg::grid_cover((hi - lo + 255) / 256, &grid, "dpg_allgather_params");
    if (st != DPG_OK) return st;
    dpg::k_allgather<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(master, va, lo, hi);
    return dpg::after_launch("dpg_allgather_params");
}

int dpg_gather_params_bf16(const dpg_plan_t* plan, const void* param_bf16, void* const* views,
                           int32_t n_views, int32_t b0, int32_t b1, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_gather_params_bf16");
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "dpg_gather_params_bf16: plan is NULL");
    const dpg::Plan& p = plan->p;
    if (b0 < 0 || b1 < b0 || b1 > p.n_buckets)
        return fail(DPG_ERR_INVALID_ARG, "dpg_gather_params_bf16: bucket range [%d, %d) outside [0, %d]",
                    b0, b1, p.n_buckets);
    if (n_views < 0 || n_views > DPG_MAX_VIEWS)
        return fail(DPG_ERR_INVALID_ARG, "dpg_gather_params_bf16: n_views %d outside [0, %d]", n_views,
                    DPG_MAX_VIEWS);
    if (b0 == b1 || n_views == 0 || p.bucket_offset[b1] == p.bucket_offset[b0]) return DPG_OK;
    if (!param_bf16) return fail(DPG_ERR_INVALID_ARG, "dpg_gather_params_bf16: param is NULL");
    if (!dpg::aligned(param_bf16, 16))
        return fail(DPG_ERR_MISALIGNED, "dpg_gather_params_bf16: param misaligned");
    if (!views) return fail(DPG_ERR_INVALID_ARG, "dpg_gather_params_bf16: views is NULL");
    dpg::ViewArgs va{};
    va.n_views = n_views;
    for (int k = 0; k < n_views; ++k) {
        if (!views[k]) return fail(DPG_ERR_INVALID_ARG, "dpg_gather_params_bf16: views[%d] is NULL", k);
        if (!dpg::aligned(views[k], 16))
            return fail(DPG_ERR_MISALIGNED, "dpg_gather_params_bf16: views[%d] misaligned", k);
        va.views[k] = views[k];
    }
    const int64_t lo = p.bucket_offset[b0] / dpg::kVec, hi = p.bucket_offset[b1] / dpg::kVec;
    int grid = 0;
    int st = dpg::grid_cover((hi - lo + 255) / 256, &grid, "dpg_gather_params_bf16");
    if (st != DPG_OK) return st;
    dpg::k_gather_bf16<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(param_bf16), va, lo, hi);
    return dpg::after_launch("dpg_gather_params_bf16");
}

static int pack_common(const dpg_plan_t* plan, const void* const* ptrs, void* flat, int unpack,
                       void* stream, const char* who) {
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "%s: plan is NULL", who);
    dpg::Plan& p = const_cast<dpg_plan_t*>(plan)->p;
    if (!flat && p.total_padded > 0) return fail(DPG_ERR_INVALID_ARG, "%s: flat buffer is NULL", who);
    if (!dpg::aligned(flat, 16)) return fail(DPG_ERR_MISALIGNED, "%s: flat buffer misaligned", who);
    if (p.n_params > 0 && !ptrs) return fail(DPG_ERR_INVALID_ARG, "%s: gradient table is NULL", who);
    for (int32_t q = 0; q < p.n_params; ++q) {
        if (p.numels[q] > 0 && !ptrs[q]) return fail(DPG_ERR_INVALID_ARG, "%s: gradient %d is NULL", who, q);
        if (!dpg::aligned(ptrs[q], 2)) return fail(DPG_ERR_MISALIGNED, "%s: gradient %d misaligned", who, q);
    }
    if (p.items.empty()) return DPG_OK;
    int st = dpg::upload(p);
    if (st != DPG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // items are in descending parameter order; launch one window of
    // kPackPtrs parameters at a time
    size_t i0 = 0;
    while (i0 < p.items.size()) {
        const int32_t top = p.items[i0].param;
        const int32_t base = top - dpg::kPackPtrs + 1 > 0 ? top - dpg::kPackPtrs + 1 : 0;
        size_t i1 = i0;
        while (i1 < p.items.size() && p.items[i1].param >= base) ++i1;
        dpg::PackArgs a{};
        for (int32_t q = base; q <= top; ++q) a.ptrs[q - base] = ptrs[q];
        a.p_base = base;
        a.unpack = unpack;
        a.items = p.d_items;
        a.item0 = int64_t(i0);
        a.flat = static_cast<uint16_t*>(flat);
        a.n_items = int64_t(i1 - i0);
        int grid = 0;
        st = dpg::grid_cover(a.n_items, &grid, who);
        if (st != DPG_OK) return st;
        dpg::k_pack<<<grid, 256, 0, s>>>(a);
        st = dpg::after_launch(who);
        if (st != DPG_OK) return st;
        i0 = i1;
    }
    return DPG_OK;
}

static int state_common(const dpg_plan_t* plan, const float* const* src, float* const* dst,
                        int32_t n_arrays, int to_flat, void* stream, const char* who) {
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "%s: plan is NULL", who);
    dpg::Plan& p = const_cast<dpg_plan_t*>(plan)->p;
    if (n_arrays < 1 || n_arrays > DPG_MAX_STATE_ARRAYS)
        return fail(DPG_ERR_INVALID_ARG, "%s: n_arrays %d outside [1, %d]", who, n_arrays,
                    DPG_MAX_STATE_ARRAYS);
    if (!src || !dst) return fail(DPG_ERR_INVALID_ARG, "%s: array table is NULL", who);
    if (p.items.empty() || p.total_padded == 0) return DPG_OK;
    dpg::StateArgs a{};
    for (int k = 0; k < n_arrays; ++k) {
        const void* flat = to_flat ? static_cast<const void*>(dst[k]) : static_cast<const void*>(src[k]);
        const void* canon = to_flat ? static_cast<const void*>(src[k]) : static_cast<const void*>(dst[k]);
        if (!flat || (!canon && p.canon_total > 0))
            return fail(DPG_ERR_INVALID_ARG, "%s: array %d is NULL", who, k);
        if (!dpg::aligned(flat, 32) || !dpg::aligned(canon, 4))
            return fail(DPG_ERR_MISALIGNED, "%s: array %d misaligned", who, k);
        a.src[k] = src[k];
        a.dst[k] = dst[k];
    }
    a.n_arrays = n_arrays;
    a.to_flat = to_flat;
    int st = dpg::upload(p);
    if (st != DPG_OK) return st;
    a.items = p.d_items;
    a.n_items = int64_t(p.items.size());
    int grid = 0;
    st = dpg::grid_cover(a.n_items, &grid, who);
    if (st != DPG_OK) return st;
    dpg::k_state_copy<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return dpg::after_launch(who);
}

int dpg_export_state(const dpg_plan_t* plan, const float* const* flat, float* const* canon,
                     int32_t n_arrays, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_export_state");
    return state_common(plan, flat, canon, n_arrays, 0, stream, "dpg_export_state");
}

int dpg_import_state(const dpg_plan_t* plan, const float* const* canon, float* const* flat,
                     int32_t n_arrays, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_import_state");
    return state_common(plan, canon, flat, n_arrays, 1, stream, "dpg_import_state");
}

int dpg_pack(const dpg_plan_t* plan, const void* const* param_grads, void* flat_bf16, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_pack");
    return pack_common(plan, param_grads, flat_bf16, 0, stream, "dpg_pack");
}

int dpg_unpack(const dpg_plan_t* plan, const void* flat_bf16, void* const* param_grads, void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_unpack");
    return pack_common(plan, const_cast<const void* const*>(param_grads), const_cast<void*>(flat_bf16),
                       1, stream, "dpg_unpack");
}

}  // extern "C"

// ---------------------------------------------------------------------------
// dpg_step_noalloc: the same fused pass and finalize, with the bucket tables
// and the norm partials in one static device array instead of memory the plan
// allocates.  For callers whose device memory the library must not allocate.
// ---------------------------------------------------------------------------
namespace dpg {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DPG_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on device `dev` (current), looked up
// once per device: in host code the symbol's name is only a host-side stand-in.
static int noalloc_scratch(int dev, unsigned char** out) {
    static std::mutex mu;
    static std::map<int, unsigned char*> addr;
    std::lock_guard<std::mutex> g(mu);
    auto it = addr.find(dev);
    if (it == addr.end()) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return fail(DPG_ERR_CUDA, "dpg_step_noalloc: cudaGetSymbolAddress failed on device %d: %s",
                        dev, cudaGetErrorString(e));
        it = addr.emplace(dev, static_cast<unsigned char*>(ptr)).first;
    }
    *out = it->second;
    return DPG_OK;
}

static int step_noalloc(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                        const void* const* last, const int64_t* tokens, int32_t n_counts,
                        const dpg_hparams* hp, float* master, float* m, float* v,
                        void* const* views, int32_t n_views, float* sqnorm, int64_t* nonfinite,
                        void* stream) {
    const char* who = "dpg_step_noalloc";
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "%s: plan is NULL", who);
    const Plan& p = plan->p;
    if (grads_dtype != DPG_BF16 && grads_dtype != DPG_F32)
        return fail(DPG_ERR_INVALID_ARG, "%s: grads_dtype %d unknown", who, grads_dtype);
    if (last && grads_dtype != DPG_F32)
        return fail(DPG_ERR_INVALID_ARG, "%s: last_micro_bf16 needs fp32 accumulation grads", who);
    if (n_views < 0 || n_views > DPG_MAX_VIEWS)
        return fail(DPG_ERR_INVALID_ARG, "%s: n_views %d outside [0, %d]", who, n_views, DPG_MAX_VIEWS);
    RsAdamArgs a{};
    int st = adam_constants(hp, a);
    if (st != DPG_OK) return st;
    st = token_scale(tokens, n_counts, &a.scale);
    if (st != DPG_OK) return st;
    if (p.n_buckets == 0) return DPG_OK;
    const bool want_norm = sqnorm || nonfinite;
    const bool has_elems = p.total_padded > 0;
    if (!has_elems && !want_norm) return DPG_OK;
    if (!has_elems) n_views = 0;

    // launch geometry, then the bytes of the static array it needs: the two
    // bucket tables and, for a norm, the visit partials of this launch
    const int mode = grads_dtype == DPG_BF16 ? kInBf16 : (last ? kInF32PlusBf16 : kInF32);
    RsKernel fn = mode == kInBf16 ? pick_rs_kernel<kInBf16>(p.R)
                : mode == kInF32 ? pick_rs_kernel<kInF32>(p.R)
                                 : pick_rs_kernel<kInF32PlusBf16>(p.R);
    int dev = 0;
    DPG_CUDA_TRY(cudaGetDevice(&dev));
    int grid = 0;
    st = fused_geometry(fn, dev, 0, p.n_tiles, 0, p.n_buckets, &grid, &a.vmax);
    if (st != DPG_OK) return st;
    const size_t nb1 = size_t(p.n_buckets) + 1;
    const size_t tab_bytes = round256(nb1 * sizeof(int64_t));
    const VisLayout L = want_norm ? vis_layout(int64_t(grid) * a.vmax, grid) : vis_layout(0, 0);
    const size_t need = 2 * tab_bytes + L.total;
    if (need > size_t(DPG_NOALLOC_SCRATCH_BYTES))
        return fail(DPG_ERR_INVALID_ARG,
                    "%s: this plan (%d buckets, %lld tiles, %d CTAs x %d bucket visits) needs %zu "
                    "bytes of scratch; the library's static scratch holds %zu bytes (use dpg_step)",
                    who, p.n_buckets, (long long)p.n_tiles, grid, a.vmax, need,
                    size_t(DPG_NOALLOC_SCRATCH_BYTES));

    if (has_elems && !grads) return fail(DPG_ERR_INVALID_ARG, "%s: grads is NULL", who);
    if (has_elems && (!master || !m || !v))
        return fail(DPG_ERR_INVALID_ARG, "%s: master/m/v must not be NULL", who);
    if (n_views > 0 && !views) return fail(DPG_ERR_INVALID_ARG, "%s: param_views is NULL", who);
    const uintptr_t galign = grads_dtype == DPG_BF16 ? 16 : 32;
    for (int r = 0; has_elems && r < p.R; ++r) {
        if (!grads[r]) return fail(DPG_ERR_INVALID_ARG, "%s: grads[%d] is NULL", who, r);
        if (!aligned(grads[r], galign)) return fail(DPG_ERR_MISALIGNED, "%s: grads[%d] misaligned", who, r);
        a.grads[r] = grads[r];
        if (last) {
            if (!last[r]) return fail(DPG_ERR_INVALID_ARG, "%s: last_micro_bf16[%d] is NULL", who, r);
            if (!aligned(last[r], 16)) return fail(DPG_ERR_MISALIGNED, "%s: last_micro_bf16[%d] misaligned", who, r);
            a.last[r] = last[r];
        }
    }
    for (int k = 0; k < n_views; ++k) {
        if (!views[k]) return fail(DPG_ERR_INVALID_ARG, "%s: param_views[%d] is NULL", who, k);
        if (!aligned(views[k], 16)) return fail(DPG_ERR_MISALIGNED, "%s: param_views[%d] misaligned", who, k);
        a.views[k] = views[k];
    }
    if (!aligned(master, 32) || !aligned(m, 32) || !aligned(v, 32))
        return fail(DPG_ERR_MISALIGNED, "%s: fp32 buffers must be 32-byte aligned", who);

    unsigned char* base = nullptr;
    st = noalloc_scratch(dev, &base);
    if (st != DPG_OK) return st;
    int64_t* d_bucket_offset = reinterpret_cast<int64_t*>(base);
    int64_t* d_tile_begin = reinterpret_cast<int64_t*>(base + tab_bytes);
    unsigned char* vis = base + 2 * tab_bytes;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the tables of this plan, in stream order ahead of the kernels that read them
    DPG_CUDA_TRY(cudaMemcpyAsync(d_bucket_offset, p.bucket_offset.data(), nb1 * sizeof(int64_t),
                                 cudaMemcpyHostToDevice, s));
    DPG_CUDA_TRY(cudaMemcpyAsync(d_tile_begin, p.tile_begin.data(), nb1 * sizeof(int64_t),
                                 cudaMemcpyHostToDevice, s));
    a.master = master;
    a.m = m;
    a.v = v;
    a.reduced = nullptr;
    a.bucket_offset = d_bucket_offset;
    a.tile_begin = d_tile_begin;
    a.t0 = 0;
    a.t1 = p.n_tiles;
    a.b0 = 0;
    a.b1 = p.n_buckets;
    a.R = p.R;
    a.n_views = n_views;
    if (want_norm) {
        a.vis_sq = reinterpret_cast<double*>(vis + L.sq);
        a.vis_nf = reinterpret_cast<int32_t*>(vis + L.nf);
        a.vis_bucket = reinterpret_cast<int32_t*>(vis + L.bucket);
        a.vis_count = reinterpret_cast<int32_t*>(vis + L.count);
    }
    return launch_fused(fn, a, grid, sqnorm, nonfinite, s, who);
}

}  // namespace dpg

extern "C" int dpg_step_noalloc(const dpg_plan_t* plan, const void* const* grads,
                                int32_t grads_dtype, const void* const* last_micro_bf16,
                                const int64_t* valid_tokens, int32_t n_counts,
                                const dpg_hparams* hp, float* master, float* exp_avg,
                                float* exp_avg_sq, void* const* param_views, int32_t n_views,
                                float* bucket_sqnorm, int64_t* bucket_nonfinite, void* stream) {
    dpg::clear_error();
    return dpg::step_noalloc(plan, grads, grads_dtype, last_micro_bf16, valid_tokens, n_counts, hp,
                             master, exp_avg, exp_avg_sq, param_views, n_views, bucket_sqnorm,
                             bucket_nonfinite, stream);
}
