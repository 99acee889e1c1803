// dpg_host.h -- host-side helpers shared by the translation units of libdpg.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <utility>

#include "dpg_device.cuh"

#define DPG_CUDA_TRY(call)                                                              \
    do {                                                                                \
        cudaError_t e_ = (call);                                                        \
        if (e_ != cudaSuccess)                                                          \
            return fail(DPG_ERR_CUDA, "%s: %s (%s)", __func__, cudaGetErrorString(e_),  \
                        #call);                                                         \
    } while (0)

namespace dpg {

// kernels launched by this library since it was loaded
extern std::atomic<int64_t> g_launches;
// the next fused launch of the calling thread records these events around itself
extern thread_local cudaEvent_t t_fused_start, t_fused_stop;
// test-only fault injection of the staged pass (consumed by its next launch)
extern thread_local int64_t t_staged_skip;
extern thread_local int64_t t_staged_timeout_ns;
// Upper bound on the CTAs of the fused passes launched from this thread (0:
// the default chunked launch; > 0 selects the persistent grid-stride kernels).
extern thread_local int32_t t_fused_max_ctas;
// 1: the streaming and chunked kernels are launched with programmatic stream
// serialization (the default); 0: plain stream-ordered launches.
extern thread_local int32_t t_programmatic;
// Checking builds: the element bound the index checks of the next launches
// from this thread use (< 0: the plan's total; a smaller bound is a test of
// the checks themselves).
extern thread_local int64_t t_debug_limit;

int sm_count(int dev, int* out);
// one CTA per unit of work (the streaming kernels)
int grid_cover(int64_t work_ctas, int* grid, const char* who);
// persistent-grid size: SM count x resident CTAs of `fn`, at most work_ctas
int grid_for(const void* fn, int threads, int dev, int64_t work_ctas, int* grid);
bool aligned(const void* p, uintptr_t a);
// checks the launch just issued and counts it
int after_launch(const char* what);
size_t round256(size_t x);

// Launches kernel k (which must begin with pdl_enter()) on `grid` CTAs of
// `block` threads, with programmatic stream serialization unless the calling
// thread switched it off, then checks and counts the launch like
// after_launch().
template <typename... P, typename... A>
int launch_k(void (*k)(P...), unsigned grid, unsigned block, cudaStream_t s, const char* who,
             A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = t_programmatic ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k, std::forward<A>(args)...);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return fail(DPG_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
    }
    return after_launch(who);
}

// Byte layout of a norm scratch with `visits` (CTA, bucket visit) slots for up
// to `ctas` CTAs; every section starts on a 256-byte boundary.
struct VisLayout {
    size_t sq, nf, bucket, count, total;
};

VisLayout vis_layout(int64_t visits, int64_t ctas);

// fp32 Adam constants (each computed in double and rounded once) into `a`
int adam_constants(const dpg_hparams* hp, RsAdamArgs& a);
// fp32(1/G) from the valid-token counts; DPG_ERR_ZERO_TOKENS when G == 0
int token_scale(const int64_t* tokens, int32_t n, float* scale);
// validates the per-call buffers of a whole-plan step and copies them into `a`
int fill_step_args(const Plan& p, const void* const* grads, int32_t grads_dtype,
                   const void* const* last, const dpg_hparams* hp, const int64_t* tokens,
                   int32_t n_counts, float* master, float* m, float* v, void* const* views,
                   int32_t n_views, RsAdamArgs& a, const char* who);
// per-bucket norms of a persistent launch of n_cta CTAs from the visit partials in `a`
int launch_norm_finalize(const RsAdamArgs& a, int32_t n_cta, int32_t n_buckets, float* sqnorm,
                         int64_t* nonfinite, cudaStream_t s, const char* who);

}  // namespace dpg
