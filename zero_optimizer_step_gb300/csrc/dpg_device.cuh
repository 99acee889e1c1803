// dpg_device.cuh -- device-side pieces shared by the kernels of libdpg.
//
// Everything on the path is a stream of HBM traffic with a few dozen ALU
// operations per element: one thread owns one 8-element vector (128-bit loads
// of every bf16 replica gradient, 256-bit loads and stores of the fp32
// master/m/v state).  The update uses the IEEE round-to-nearest intrinsics
// (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn, __fsub_rn), which the
// compiler never contracts into FMAs, in the order of Kingma & Ba's
// Algorithm 1, so the results are the oracle's bits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dpg_internal.h"

namespace dpg {

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
// Deferred accumulation: K bf16 microbatch buffers per replica, replica-major
// (grads[r * K + k]); MODE = kInBf16Deferred + KT, KT = K fixed at compile
// time, or 0 for K read from the arguments.
constexpr int kInBf16Deferred = 16;

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
    int32_t K;           // deferred accumulation: microbatches per replica
    float scale;         // fp32(1/G)
    float beta1, beta2, omb1, omb2, bias1, bias2, lr, eps, lr_wd;
    int32_t decay;
    const float* g_in;      // kInReduced: the normalised reduced gradient
    const float* clip_coef; // kUpdate: device scalar, g <- g * coef
    // chunked launches (one CTA per chunk): per tile {first element, end of
    // its bucket} and the per-chunk norm partials (NULL: no norm)
    const longlong2* tile_span;
    double* chunk_sq;
    int32_t* chunk_nf;
#ifdef DPG_DEBUG
    unsigned long long* dbg;  // the plan's debug word (NULL: checks record nothing)
    int64_t dbg_limit;        // elements an index must stay below (the plan's total)
#endif
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
            // any R: replicas in groups of four whose loads are all issued
            // before their adds (still added in rank order)
            widen8(ld_grad_u4(static_cast<const uint16_t*>(a.grads[0]) + i), s);
            int r = 1;
            for (; r + 4 <= R; r += 4) {
                uint4 x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    x[u] = ld_grad_u4(static_cast<const uint16_t*>(a.grads[r + u]) + i);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float t[8];
                    widen8(x[u], t);
#pragma unroll
                    for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], t[j]);
                }
            }
            uint4 x[3];
            const int rem = R - r;                            // 0..3
#pragma unroll
            for (int u = 0; u < 3; ++u)
                if (u < rem) x[u] = ld_grad_u4(static_cast<const uint16_t*>(a.grads[r + u]) + i);
#pragma unroll
            for (int u = 0; u < 3; ++u) {
                if (u < rem) {
                    float t[8];
                    widen8(x[u], t);
#pragma unroll
                    for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], t[j]);
                }
            }
        }
    } else if constexpr (MODE >= kInBf16Deferred) {
        // each replica's K microbatches summed in microbatch order -- the
        // binary32 additions of the no_sync accumulation path -- then the
        // replicas in rank order
        constexpr int KT = MODE - kInBf16Deferred;
        const int K = KT > 0 ? KT : a.K;
#pragma unroll(RT > 0 ? RT : 1)
        for (int r = 0; r < R; ++r) {
            const void* const* g = a.grads + r * K;
            float x[8];
            if constexpr (KT > 0) {
                uint4 q[KT];
#pragma unroll
                for (int k = 0; k < KT; ++k) q[k] = ld_grad_u4(static_cast<const uint16_t*>(g[k]) + i);
                widen8(q[0], x);
#pragma unroll
                for (int k = 1; k < KT; ++k) {
                    float t[8];
                    widen8(q[k], t);
#pragma unroll
                    for (int j = 0; j < 8; ++j) x[j] = __fadd_rn(x[j], t[j]);
                }
            } else {
                widen8(ld_grad_u4(static_cast<const uint16_t*>(g[0]) + i), x);
                for (int k = 1; k < K; ++k) {
                    float t[8];
                    widen8(ld_grad_u4(static_cast<const uint16_t*>(g[k]) + i), t);
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

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization can be scheduled while the kernel before it in the stream is
// still draining.  griddepcontrol.wait holds every thread until that kernel
// has completed and its writes are visible (it returns at once for a plain
// launch), so nothing is read or written before it; the trigger that follows
// lets the next such kernel be scheduled in turn, to wait behind this one.
// Every kernel launched through launch_k() starts with this.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#ifdef DPG_DEBUG
// Index checks of a checking build (-DDPG_DEBUG): a table-driven kernel checks
// the element and table indices it derives from the plan's device tables
// before using them.  A failed check records (code << 32 | CTA index) as the
// first failure in the plan's debug word and the access is skipped; nothing
// traps, and control flow (barriers) is unchanged.  Codes: 1 chunked fused or
// norm pass, 2 chunk finalize (long buckets), 3 chunk finalize (short
// buckets), 4 pack / unpack.
__device__ __forceinline__ bool debug_ok(unsigned long long* word, bool ok, unsigned code) {
    if (!ok && word != nullptr)
        atomicCAS(word, 0ull, (static_cast<unsigned long long>(code) << 32) | blockIdx.x);
    return ok;
}
#endif

// Chunked launches: one 128-thread CTA per 1024-element chunk (a quarter of a
// bucket-aligned tile), one 8-element vector per thread.
constexpr int kChunkThreads = 128;
constexpr int kChunk = kChunkThreads * kVec;
constexpr int kChunksPerTile = int(kTile / kChunk);

}  // namespace dpg
