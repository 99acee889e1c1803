// dpg_stream.cu -- the streaming kernels around the fused pass: no_sync
// accumulation (single and paired), the fp32 -> bf16 all-gather, the ZeRO-3
// bf16 gather, pack/unpack of parameter-shaped gradients, and the optimizer
// state's checkpoint layout conversions.  Each launches one CTA per unit of
// work.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dpg_host.h"

namespace dpg {

// ---------------------------------------------------------------------------
// no_sync accumulation and the stand-alone all-gather
// ---------------------------------------------------------------------------
template <bool FIRST>
__global__ void __launch_bounds__(256) k_accumulate(const uint16_t* __restrict__ g,
                                                    float* __restrict__ acc, int64_t n_vec) {
    pdl_enter();
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
    pdl_enter();
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
    pdl_enter();
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
    pdl_enter();
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
#ifdef DPG_DEBUG
    unsigned long long* dbg;  // the plan's debug word
    int64_t dbg_limit;        // elements of the flat buffer
#endif
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

// CTA c copies item c of the launch's window (launched with one CTA per item;
// the loop also serves a smaller grid).
__global__ void __launch_bounds__(256) k_pack(const __grid_constant__ PackArgs a) {
    for (int64_t j = blockIdx.x; j < a.n_items; j += gridDim.x) {
        const PackItem it = a.items[a.item0 + j];
#ifdef DPG_DEBUG
        if (!debug_ok(a.dbg, it.param - a.p_base >= 0 && it.param - a.p_base < kPackPtrs &&
                                 it.flat_off >= 0 && it.count >= 0 && it.tail >= 0 &&
                                 it.src_off >= 0 &&
                                 it.flat_off + it.count + (a.unpack ? 0 : it.tail) <= a.dbg_limit,
                      4))
            continue;                           // uniform over the CTA: no barrier below
#endif
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
// registration-order layout, one CTA per item
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

}  // namespace dpg

using dpg::fail;

extern "C" {

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
    return dpg::launch_k(first ? dpg::k_accumulate<true> : dpg::k_accumulate<false>, grid, 256, s,
                         "dpg_accumulate", g, acc_f32, n_vec);
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
    return dpg::launch_k(first ? dpg::k_accumulate_pair<true> : dpg::k_accumulate_pair<false>, grid,
                         256, s, "dpg_accumulate_pair", ga, gb, acc_f32, n_vec);
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
    return dpg::launch_k(dpg::k_allgather, grid, 256, static_cast<cudaStream_t>(stream),
                         "dpg_allgather_params", master, va, lo, hi);
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
    return dpg::launch_k(dpg::k_gather_bf16, grid, 256, static_cast<cudaStream_t>(stream),
                         "dpg_gather_params_bf16", static_cast<const uint16_t*>(param_bf16), va, lo,
                         hi);
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
#ifdef DPG_DEBUG
        a.dbg = p.d_debug;
        a.dbg_limit = dpg::t_debug_limit >= 0 ? dpg::t_debug_limit : p.total_padded;
#endif
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
