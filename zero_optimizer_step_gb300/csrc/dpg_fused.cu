// dpg_fused.cu -- the fused reduce-scatter + normalisation + Adam + bf16
// all-gather pass and its variants: the chunked kernels (one small CTA per
// 1024-element chunk, the default), the persistent grid-stride kernels (a
// grid cap, the allocation-free step, the clipped norm pass over R <= 4
// re-read replicas), the clipped step's norm pass, the per-bucket norm
// finalizes, and their C entry points.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>

#include "dpg_host.h"

namespace dpg {

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
    pdl_enter();
    const int64_t c = blockIdx.x;                         // chunk of this launch
    const longlong2 span = __ldg(a.tile_span + a.t0 + c / kChunksPerTile);
    const int64_t i = span.x + (c % kChunksPerTile) * kChunk + int64_t(threadIdx.x) * kVec;
    float sq = 0.0f;
    int nf = 0;
#ifdef DPG_DEBUG
    const bool in_range = debug_ok(a.dbg, span.x >= 0 && span.x <= span.y && span.y <= a.dbg_limit &&
                                              (i >= span.y || i + kVec <= span.y), 1);
#else
    constexpr bool in_range = true;
#endif
    if (i < span.y && in_range) {
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
        constexpr int W = kChunkThreads / 32;
        __shared__ double w_sq[W];
        __shared__ int w_nf[W];
        const int warp = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0) {
            w_sq[warp] = double(sq);
            w_nf[warp] = nf;
        }
        // Warps 1..W-1 only signal named barrier 1 (its arrive orders their
        // slot writes before warp 0's reads) and retire; warp 0 waits for all
        // kChunkThreads arrivals and sums the slots in warp order.  Every
        // thread of the CTA reaches exactly one of the two instructions.
        if (warp != 0) {
            asm volatile("bar.arrive 1, %0;" ::"n"(kChunkThreads) : "memory");
        } else {
            asm volatile("bar.sync 1, %0;" ::"n"(kChunkThreads) : "memory");
            if (threadIdx.x == 0) {
                double tot = 0.0;
                int cnt = 0;
#pragma unroll
                for (int k = 0; k < W; ++k) {
                    tot += w_sq[k];
                    cnt += w_nf[k];
                }
                a.chunk_sq[c] = tot;
                a.chunk_nf[c] = cnt;
            }
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
    pdl_enter();
    const int64_t c = blockIdx.x;
    const longlong2 span = __ldg(a.tile_span + a.t0 + c / CPT);
    const int64_t i = span.x + (c % CPT) * CH + int64_t(threadIdx.x) * kVec;
    const bool norm = a.chunk_sq != nullptr;
    NormAcc acc;
    int nf = 0;
#ifdef DPG_DEBUG
    const bool in_range = debug_ok(a.dbg, span.x >= 0 && span.x <= span.y && span.y <= a.dbg_limit &&
                                              (i >= span.y || i + kVec <= span.y), 1);
#else
    constexpr bool in_range = true;
#endif
    if (i < span.y && in_range) {
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

// Per-bucket norms of a chunked launch from its per-chunk partials.  One CTA
// per segment (at most kSegTiles tiles of one bucket): thread j adds the
// segment's chunks j + 1024 k in increasing k, 8 loads in flight, then a fixed
// butterfly tree (within each warp, then over the 32 warp sums) gives the
// segment's sum.  The CTA that completes a bucket's last segment (a per-bucket
// arrival counter, which it resets to zero for the next launch) adds the
// bucket's segment sums in segment order.  A short bucket (at most
// kShortTiles tiles: one segment of <= 1024 chunks) is summed by one warp
// along the same tree, so it gets the same bits.
// One launch does both: the long buckets' segment CTAs first, then CTAs of
// 32 warps for the short buckets.  Every grouping is fixed by the plan, so
// the result is the same on every run and for any bucket range.
constexpr int kChunkFinalizeThreads = 1024;
static_assert(kShortTiles * kChunksPerTile <= kChunkFinalizeThreads && kShortTiles <= kSegTiles,
              "a short bucket is one segment with at most one chunk per finalize thread");

struct FinalizeArgs {
    const double* chunk_sq;     // per-chunk partials of the launch (chunk 0 = tile t0)
    const int32_t* chunk_nf;
    const int64_t* tile_begin;  // plan tables
    const int32_t* seg_first;
    const int32_t* seg_bucket;
    double* seg_sq;             // per-segment sums
    long long* seg_nf;
    int32_t* done;              // per-bucket arrival counters
    const int32_t* long_list;   // segment ids of the long buckets
    const int32_t* short_list;  // short bucket ids
    int64_t t0;                 // first tile of the launch
    int32_t cpt;                // chunks per tile
    int32_t l0, l1;             // the launch's slice of long_list
    int32_t q0, q1;             // the launch's slice of short_list
    int32_t short_per_cta;      // short buckets (warps) per CTA, <= 32
#ifdef DPG_DEBUG
    unsigned long long* dbg;    // the plan's debug word
    int64_t dbg_chunks;         // chunk partials of the launch
    int32_t dbg_buckets, dbg_segs;
#endif
    float* sqnorm;              // outputs, indexed by bucket (nullable)
    int64_t* nonfinite;
    double* sqnorm64;
};

// One warp per short bucket (n <= 1024 chunks, a single segment): the same
// tree as k_chunk_finalize.  There thread j of the segment's CTA holds
// 0 + chunk j (chunk j < n; 0 otherwise; adding zeros to a non-negative sum
// of squares changes nothing), each warp sums its 32 threads by butterfly,
// and warp 0 sums the 32 warp results by butterfly; here the warp forms the
// 32 warp results one after the other, lane w keeping the w-th, then sums
// them by the same butterfly.
__device__ __forceinline__ void finalize_short_bucket(const FinalizeArgs& f, int32_t q) {
    constexpr int U = 8;
    const int lane = threadIdx.x & 31;
    if (q >= f.q1) return;
    const int b = __ldg(f.short_list + q);
#ifdef DPG_DEBUG
    if (!debug_ok(f.dbg, b >= 0 && b < f.dbg_buckets, 3)) return;   // warp-uniform
#endif
    const int64_t cb = (__ldg(f.tile_begin + b) - f.t0) * f.cpt;
    int n = int((__ldg(f.tile_begin + b + 1) - f.t0) * f.cpt - cb);
#ifdef DPG_DEBUG
    // a failed check: no partial is loaded and the bucket's outputs are not written
    const bool bad = !debug_ok(f.dbg, cb >= 0 && n >= 0 && n <= 1024 && cb + n <= f.dbg_chunks, 3);
    if (bad) n = 0;
#endif
    const int rows = (n + 31) >> 5;       // warp results with any chunk (<= 32)
    double keep = 0.0;
    long long keep_n = 0;
    for (int w0 = 0; w0 < rows; w0 += U) {
        double x[U];
        int y[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int k = (w0 + u) * 32 + lane;
            x[u] = k < n ? f.chunk_sq[cb + k] : 0.0;
            y[u] = k < n ? f.chunk_nf[cb + k] : 0;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (w0 + u >= rows) break;        // the rest are sums of zeros: 0 (uniform)
            double acc = 0.0;
            long long cnt = 0;
            acc += x[u];
            cnt += y[u];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
                cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
            }
            if (lane == w0 + u) {
                keep = acc;
                keep_n = cnt;
            }
        }
    }
    // with one warp result (n <= 32) the tree over the 32 results adds only
    // zeros to it, which changes no bit of a sum of squares
    if (rows > 1) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            keep += __shfl_xor_sync(0xFFFFFFFFu, keep, o);
            keep_n += __shfl_xor_sync(0xFFFFFFFFu, keep_n, o);
        }
    }
    if (lane != 0) return;
#ifdef DPG_DEBUG
    if (bad) return;
#endif
    // the CTA path's last step adds the bucket's one segment sum to 0.0
    double tot = 0.0;
    tot += keep;
    if (f.sqnorm) f.sqnorm[b] = float(tot);
    if (f.nonfinite) f.nonfinite[b] = keep_n;
    if (f.sqnorm64) f.sqnorm64[b] = tot;
}

__global__ void __launch_bounds__(kChunkFinalizeThreads)
k_chunk_finalize(const __grid_constant__ FinalizeArgs f) {
    constexpr int T = kChunkFinalizeThreads, U = 8, NW = T / 32;
    static_assert(NW == 32, "warp 0 combines one sum per warp, one per lane");
    __shared__ double w_sq[NW];
    __shared__ long long w_nf[NW];
    pdl_enter();
    // CTAs [0, l1 - l0): one long-bucket segment each; the CTAs after them:
    // one short bucket per warp
    const int32_t n_long = f.l1 - f.l0;
    if (int32_t(blockIdx.x) >= n_long) {
        const int32_t warp = int32_t(threadIdx.x >> 5);
        if (warp < f.short_per_cta)
            finalize_short_bucket(f, f.q0 + (int32_t(blockIdx.x) - n_long) * f.short_per_cta + warp);
        return;
    }
    int32_t s = __ldg(f.long_list + f.l0 + int32_t(blockIdx.x));
#ifdef DPG_DEBUG
    // a failed check: the table reads stay at index 0, the CTA loads no
    // partial and writes nothing (it still meets the CTA barrier)
    bool bad = !debug_ok(f.dbg, s >= 0 && s < f.dbg_segs, 2);
    if (bad) s = 0;
#endif
    int b = __ldg(f.seg_bucket + s);
#ifdef DPG_DEBUG
    if (!bad && !debug_ok(f.dbg, b >= 0 && b < f.dbg_buckets, 2)) bad = true;
    if (bad) b = 0;
#endif
    const int64_t span = kSegTiles * f.cpt;
    const int64_t cb = (__ldg(f.tile_begin + b) - f.t0) * f.cpt;
    const int64_t ce = (__ldg(f.tile_begin + b + 1) - f.t0) * f.cpt;
    const int64_t c0 = cb + int64_t(s - __ldg(f.seg_first + b)) * span;
#ifdef DPG_DEBUG
    if (!bad && !debug_ok(f.dbg, cb >= 0 && c0 >= cb && ce <= f.dbg_chunks, 2)) bad = true;
    const int64_t c1 = bad ? c0 : (c0 + span < ce ? c0 + span : ce);
#else
    const int64_t c1 = c0 + span < ce ? c0 + span : ce;
#endif
    double acc = 0.0;
    long long cnt = 0;
    for (int64_t c = c0 + threadIdx.x; c < c1; c += int64_t(T) * U) {
        double x[U];
        int y[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = c + int64_t(u) * T;
            x[u] = k < c1 ? f.chunk_sq[k] : 0.0;
            y[u] = k < c1 ? f.chunk_nf[k] : 0;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            acc += x[u];
            cnt += y[u];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        w_sq[warp] = acc;
        w_nf[warp] = cnt;
    }
    __syncthreads();
    if (warp != 0) return;
    acc = w_sq[lane];
    cnt = w_nf[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
    }
    if (lane != 0) return;
#ifdef DPG_DEBUG
    if (bad) return;
#endif
    f.seg_sq[s] = acc;
    f.seg_nf[s] = cnt;
    __threadfence();                      // the sums before the arrival
    const int32_t first = __ldg(f.seg_first + b), end = __ldg(f.seg_first + b + 1);
    if (atomicAdd(f.done + b, 1) != end - first - 1) return;
    __threadfence();                      // every arrival before the reads
    double tot = 0.0;
    long long n = 0;
    for (int32_t k = first; k < end; ++k) {
        tot += __ldcg(f.seg_sq + k);
        n += __ldcg(f.seg_nf + k);
    }
    if (f.sqnorm) f.sqnorm[b] = float(tot);
    if (f.nonfinite) f.nonfinite[b] = n;
    if (f.sqnorm64) f.sqnorm64[b] = tot;
    f.done[b] = 0;                        // ready for the next launch
}

// Global clip coefficient from the per-bucket squared norms (one CTA, fixed
// order): norm = sqrt(sum), coef = min(1, max_norm / (norm + 1e-6)) in double,
// stored as fp32; a NaN norm gives a NaN coefficient (it is not clamped away).
__global__ void __launch_bounds__(256) k_clip_coef(const double* __restrict__ bucket_sq, int32_t nb,
                                                   double max_norm, float* coef, float* out) {
    __shared__ double sh[256];
    pdl_enter();
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
    a.tile_span = reinterpret_cast<const longlong2*>(p.d_tile_span);
    a.chunk_sq = want_norm ? p.d_chunk_sq : nullptr;
    a.chunk_nf = want_norm ? p.d_chunk_nf : nullptr;
#ifdef DPG_DEBUG
    a.dbg = p.d_debug;
    a.dbg_limit = t_debug_limit >= 0 ? t_debug_limit : p.total_padded;
#endif
    const int64_t n_chunks = (a.t1 - a.t0) * cpt;
    if (n_chunks > 0x7FFFFFFF) return fail(DPG_ERR_INVALID_ARG, "%s: %lld chunks in one launch", who,
                                           (long long)n_chunks);
    int st = DPG_OK;
    if (n_chunks > 0) {
        cudaEvent_t ev0 = t_fused_start, ev1 = t_fused_stop;
        t_fused_start = t_fused_stop = nullptr;
        if (ev0) DPG_CUDA_TRY(cudaEventRecord(ev0, s));
        st = launch_k(fn, unsigned(n_chunks), threads, s, who, a);
        if (st != DPG_OK) return st;
        if (ev1) DPG_CUDA_TRY(cudaEventRecord(ev1, s));
    }
    if (want_norm) {
        FinalizeArgs f{};
        f.chunk_sq = p.d_chunk_sq;
        f.chunk_nf = p.d_chunk_nf;
        f.tile_begin = p.d_tile_begin;
        f.seg_first = p.d_seg_first;
        f.seg_bucket = p.d_seg_bucket;
        f.seg_sq = p.d_seg_sq;
        f.seg_nf = p.d_seg_nf;
        f.done = p.d_bucket_done;
        f.t0 = a.t0;
        f.cpt = cpt;
        f.sqnorm = sqnorm;
        f.nonfinite = nonfinite;
        f.sqnorm64 = sqnorm64;
#ifdef DPG_DEBUG
        f.dbg = p.d_debug;
        f.dbg_chunks = n_chunks;
        f.dbg_buckets = p.n_buckets;
        f.dbg_segs = p.n_seg;
#endif
        // the range's long-bucket segments (one CTA each), then its short
        // buckets (one warp each)
        f.long_list = p.d_long_seg;
        f.l0 = p.long_first[size_t(a.b0)];
        f.l1 = p.long_first[size_t(a.b1)];
        f.short_list = p.d_short_bucket;
        f.q0 = p.short_first[size_t(a.b0)];
        f.q1 = p.short_first[size_t(a.b1)];
        // the short buckets are spread over the SMs: up to 32 warps per CTA,
        // fewer when there are fewer short buckets than 32 per SM
        int sms = 1;
        st = sm_count(p.device, &sms);
        if (st != DPG_OK) return st;
        const int32_t n_short = f.q1 - f.q0;
        int32_t per = (n_short + sms - 1) / sms;
        per = per < 1 ? 1 : (per > kChunkFinalizeThreads / 32 ? kChunkFinalizeThreads / 32 : per);
        f.short_per_cta = per;
        const int64_t grid = int64_t(f.l1 - f.l0) + (n_short + per - 1) / per;
        if (grid > 0) st = launch_k(k_chunk_finalize, unsigned(grid), kChunkFinalizeThreads, s, who, f);
    }
    return st;
}

static int rs_adam(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                   const void* const* last, const int64_t* tokens, int32_t n_counts,
                   const dpg_hparams* hp, float* master, float* m, float* v,
                   void* const* views, int32_t n_views, float* sqnorm, int64_t* nonfinite,
                   float* reduced, int32_t b0, int32_t b1, void* stream, const char* who,
                   const void* const* last2 = nullptr, bool check_only = false) {
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
    if (st != DPG_OK || check_only) return st;

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
int fill_step_args(const Plan& p, const void* const* grads, int32_t grads_dtype,
                   const void* const* last, const dpg_hparams* hp, const int64_t* tokens,
                   int32_t n_counts, float* master, float* m, float* v, void* const* views,
                   int32_t n_views, RsAdamArgs& a, const char* who) {
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

// Whole step with deferred accumulation: every replica's K bf16 microbatch
// buffers summed inside the fused pass (see dpg_step_deferred in
// include/dpg.h).  Always the chunked launch.
static int step_deferred(const dpg_plan_t* plan, const void* const* micro, int32_t K,
                         const int64_t* tokens, int32_t n_counts, const dpg_hparams* hp,
                         float* master, float* m, float* v, void* const* views, int32_t n_views,
                         float* sqnorm, int64_t* nonfinite, void* stream) {
    const char* who = "dpg_step_deferred";
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "%s: plan is NULL", who);
    Plan& p = const_cast<dpg_plan_t*>(plan)->p;
    if (K < 1 || int64_t(K) * p.R > DPG_MAX_REPLICAS)
        return fail(DPG_ERR_INVALID_ARG, "%s: K = %d microbatches with R = %d needs 1 <= K and "
                    "R * K <= %d", who, K, p.R, DPG_MAX_REPLICAS);
    RsAdamArgs a{};
    int st = fill_step_args(p, micro, DPG_BF16, nullptr, hp, tokens, n_counts, master, m, v, views,
                            n_views, a, who);
    if (st != DPG_OK) return st;
    const bool want_norm = sqnorm || nonfinite;
    if (p.n_buckets == 0 || (p.total_padded == 0 && !want_norm)) return DPG_OK;
    for (int q = 0; p.total_padded > 0 && q < p.R * K; ++q) {
        if (!micro[q]) return fail(DPG_ERR_INVALID_ARG, "%s: microbatch buffer %d is NULL", who, q);
        if (!aligned(micro[q], 16)) return fail(DPG_ERR_MISALIGNED, "%s: microbatch buffer %d misaligned", who, q);
        a.grads[q] = micro[q];
    }
    st = upload(p);
    if (st != DPG_OK) return st;
    a.K = K;
    a.bucket_offset = p.d_bucket_offset;
    a.tile_begin = p.d_tile_begin;
    a.t0 = 0;
    a.t1 = p.n_tiles;
    a.b0 = 0;
    a.b1 = p.n_buckets;
    RsKernel fc;
    if (K == 4) {
        switch (p.R) {
            case 1: fc = k_rs_adam_chunk<1, kInBf16Deferred + 4, kFull>; break;
            case 2: fc = k_rs_adam_chunk<2, kInBf16Deferred + 4, kFull>; break;
            case 4: fc = k_rs_adam_chunk<4, kInBf16Deferred + 4, kFull>; break;
            case 8: fc = k_rs_adam_chunk<8, kInBf16Deferred + 4, kFull>; break;
            default: fc = k_rs_adam_chunk<0, kInBf16Deferred + 4, kFull>; break;
        }
    } else {
        fc = pick_chunk_kernel<kInBf16Deferred>(p.R);
    }
    return launch_chunked(fc, a, p, want_norm, sqnorm, nonfinite, static_cast<cudaStream_t>(stream),
                          who);
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
    st = launch_k(k_clip_coef, 1, 256, s, who, static_cast<const double*>(p.d_bucket_sq64),
                  p.n_buckets, max_norm, p.d_clip_coef, clip_out);
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

int launch_norm_finalize(const RsAdamArgs& a, int32_t n_cta, int32_t n_buckets, float* sqnorm,
                         int64_t* nonfinite, cudaStream_t s, const char* who) {
    k_norm_finalize<<<n_buckets, kFinalizeThreads, 0, s>>>(a.vis_sq, a.vis_nf, a.vis_bucket,
                                                          a.vis_count, n_cta, a.vmax, 0, sqnorm,
                                                          nonfinite, nullptr);
    return after_launch(who);
}

}  // namespace dpg

using dpg::fail;

extern "C" {

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

int dpg_reduce_scatter_adam_when_ready(const dpg_plan_t* plan, const void* const* grads,
                                       int32_t grads_dtype, const void* const* last_micro_bf16,
                                       const int64_t* valid_tokens, int32_t n_counts,
                                       const dpg_hparams* hp, float* master, float* exp_avg,
                                       float* exp_avg_sq, void* const* param_views,
                                       int32_t n_views, float* bucket_sqnorm,
                                       int64_t* bucket_nonfinite, float* reduced_grad, int32_t b0,
                                       int32_t b1, void* const* ready_events, void* stream) {
    dpg::clear_error();
    const char* who = "dpg_reduce_scatter_adam_when_ready";
    const dpg::Trace trace(who);
    // every argument is checked once, over the whole range, before the stream
    // is given any wait or launch
    if (!plan) return fail(DPG_ERR_INVALID_ARG, "%s: plan is NULL", who);
    if (b0 >= 0 && b1 > b0 && b1 <= plan->p.n_buckets) {
        if (!ready_events) return fail(DPG_ERR_INVALID_ARG, "%s: ready_events is NULL", who);
        for (int32_t b = b0; b < b1; ++b)
            if (!ready_events[b - b0])
                return fail(DPG_ERR_INVALID_ARG, "%s: ready_events[%d] is NULL", who, b - b0);
    }
    int st = dpg::rs_adam(plan, grads, grads_dtype, last_micro_bf16, valid_tokens, n_counts, hp,
                          master, exp_avg, exp_avg_sq, param_views, n_views, bucket_sqnorm,
                          bucket_nonfinite, reduced_grad, b0, b1, stream, who, nullptr, true);
    if (st != DPG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int32_t b = b0; b < b1; ++b) {
        DPG_CUDA_TRY(cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(ready_events[b - b0]), 0));
        st = dpg::rs_adam(plan, grads, grads_dtype, last_micro_bf16, valid_tokens, n_counts, hp,
                          master, exp_avg, exp_avg_sq, param_views, n_views, bucket_sqnorm,
                          bucket_nonfinite, reduced_grad, b, b + 1, stream, who);
        if (st != DPG_OK) return st;
    }
    return DPG_OK;
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

int dpg_step_deferred(const dpg_plan_t* plan, const void* const* micro_bf16, int32_t K,
                      const int64_t* valid_tokens, int32_t n_counts, const dpg_hparams* hp,
                      float* master, float* exp_avg, float* exp_avg_sq, void* const* param_views,
                      int32_t n_views, float* bucket_sqnorm, int64_t* bucket_nonfinite,
                      void* stream) {
    dpg::clear_error();
    const dpg::Trace trace("dpg_step_deferred");
    return dpg::step_deferred(plan, micro_bf16, K, valid_tokens, n_counts, hp, master, exp_avg,
                              exp_avg_sq, param_views, n_views, bucket_sqnorm, bucket_nonfinite,
                              stream);
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

