/*
 * dpg.h -- C ABI of the GB300 (sm_103a) data-parallel ZeRO-2 gradient step.
 *
 * The step, as the pages describe it for DDP and ZeRO-1/2:
 *   gradients are collected into byte-capped flat buckets in backward-ready
 *   (reverse) order; each bucket is reduce-scattered so that rank r owns the
 *   r-th 1/R shard of the summed gradient; the owner normalises it by the
 *   global valid-token count and applies mixed-precision Adam to its shard of
 *   fp32 master weight and moments; the updated bf16 parameters are
 *   all-gathered back to every replica.
 * Sources (page title, section):
 *   "Parallelisms" -- Data parallel; Gradient bucketing; ZeRO-1; ZeRO-2;
 *       FSDP (Flat parameter; YaFSDP writes gradients into comm buffers).
 *   "Distributed Training and Parallelism" -- Data parallelism and the global
 *       gradient (R/global_count normalisation, no_sync accumulation).
 *   "Parallelism Starts With the Bottleneck" -- Allreduce equals
 *       reducescatter plus allgather; ZeRO removes the copies.
 *   Adam itself: Kingma & Ba (2015), Algorithm 1 (the pages name it only).
 *
 * On one GPU the R data-parallel replicas are R gradient buffers resident in
 * the same HBM; the reduce-scatter is an on-device rank-ordered reduction into
 * R shards and the all-gather is a bf16 cast written to the replica views.
 *
 * Conventions for every function below
 *   - Returns DPG_OK (0) or a negative DPG_ERR_* code; dpg_last_error() then
 *     holds a message for the calling thread.  No exception crosses the ABI;
 *     nothing calls exit() or traps on the device.
 *   - The CALLER owns every device buffer passed in.  The library owns only
 *     the plan object (host tables, their device copy and the scratch used for
 *     the per-bucket norm partials), freed by dpg_plan_destroy().
 *   - "flat" buffers hold plan->total_padded elements laid out bucket after
 *     bucket (see dpg_plan_buckets).  bf16 buffers must be 16-byte aligned,
 *     fp32 buffers 32-byte aligned (DPG_ERR_MISALIGNED otherwise).
 *   - Device work is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  Host arrays passed in (pointer tables, token
 *     counts, hparams) are read before the call returns.
 *   - A plan uploads its tables to the current device on its first device
 *     call (a synchronous copy), or explicitly with dpg_plan_upload(); call
 *     that before capturing a stream into a CUDA graph.  A plan serves one
 *     device.  Calls that use the norm scratch of the same plan (its
 *     partials and per-bucket arrival counters, which every call leaves at
 *     zero) must not overlap on the GPU (issue them on one stream).
 *   - Gradient INPUTS (grads, last_micro, the accumulate sources) of
 *     dpg_accumulate, dpg_accumulate_pair, dpg_reduce_scatter_adam, dpg_step,
 *     dpg_step_fold2, dpg_step_clipped and dpg_allreduce_grads may instead be
 *     page-locked host memory
 *     (cudaHostAlloc / cudaMallocHost, or host-registered) at its own
 *     address, which unified addressing maps into the device: the kernels
 *     then read it over the host link with the same loads, so no staging
 *     copy or device gradient buffer is needed and the results are the
 *     same bits.  The pass then runs at the link's bandwidth, not HBM's.
 *     The staged and allocation-free steps take device memory only.  The
 *     library does not query pointer kinds (that would cost a driver call
 *     per pointer per launch): every other pointer must be device memory,
 *     and pageable (unregistered) host memory is not a valid input.
 */
#ifndef DPG_H
#define DPG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define DPG_OK 0
#define DPG_ERR_INVALID_ARG (-1)    /* bad pointer/size/count/dtype/range      */
#define DPG_ERR_ZERO_TOKENS (-2)    /* global valid-token count G == 0          */
#define DPG_ERR_MISALIGNED (-3)     /* a buffer breaks the alignment rule       */
#define DPG_ERR_CUDA (-4)           /* a CUDA runtime call or launch failed     */
#define DPG_ERR_DEVICE_TIMEOUT (-5) /* a bounded device-side wait gave up       */
#define DPG_ERR_OOM (-6)            /* host or device allocation of the plan    */

/* gradient buffer element types */
#define DPG_BF16 0
#define DPG_F32 1

#define DPG_MAX_REPLICAS 64 /* R */
#define DPG_MAX_VIEWS 64    /* bf16 parameter views written by one call */

typedef struct dpg_plan dpg_plan_t;

/* Adam hyper-parameters.  step = t of this update, after increment (the first
 * update uses 1).  The library rounds each constant once to fp32:
 * beta1, beta2, 1-beta1, 1-beta2, 1-beta1^t, 1-beta2^t, lr, eps, lr*wd are
 * computed in double and converted.  weight_decay != 0 applies decoupled
 * (AdamW) decay w <- w - (lr*wd)*w before the Adam update. */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    int64_t step;
} dpg_hparams;

/* Message describing the last failure on the calling thread ("" if none). */
const char* dpg_last_error(void);
/* Static name of a status code. */
const char* dpg_status_string(int status);
/* ABI version of this header (bumped on any signature change). */
int dpg_abi_version(void);
#define DPG_ABI_VERSION 1

/* ---------------------------------------------------------------------------
 * Bucket plan (host)                ["Parallelisms" -- Data parallel; Gradient
 *                                    bucketing; ZeRO-2; FSDP / Flat parameter]
 * numels[n_params]: element counts in module REGISTRATION order (>= 0).
 * Parameters are placed in REVERSE order (later layers are ready first in
 * backward).  Each slice starts on a multiple of 8 elements.  A parameter with
 * elements that would take a bucket already holding elements past cap_bytes
 * (2 bytes per bf16 gradient element, alignment included) first closes it; a
 * parameter larger than the cap sits alone; parameters are never split;
 * zero-size parameters never close a bucket.  A closed bucket is zero-padded
 * to a multiple of 8*R elements; shard r of bucket b is
 * [r*padded_b/R, (r+1)*padded_b/R) inside it.  Buckets follow one another in
 * the flat buffer in closing order (bucket 0 holds the last parameters).
 * 1 <= R <= DPG_MAX_REPLICAS, cap_bytes > 0, n_params >= 0.  Host only: needs
 * no GPU.  *out receives a new plan (free with dpg_plan_destroy).
 * ------------------------------------------------------------------------- */
int dpg_plan_buckets(const int64_t* numels, int32_t n_params, int64_t cap_bytes,
                     int32_t R, dpg_plan_t** out);

/* Shard plan of the ZeRO-2 split across R data-parallel ranks, one GPU each
 * ["Parallelisms" -- ZeRO-2; "Parallelism Starts With the Bottleneck" --
 *  Allreduce equals reducescatter plus allgather].  Rank r owns shard r of
 * every bucket of `plan`.  *out receives a plan with the same R and one
 * bucket per bucket of `plan`: its bucket b holds one slice of
 * shard_numel_b = padded_b / R elements (the shard), zero-padded to a
 * multiple of 8*R.  It is the same for every rank.  A rank lays out by it
 * the slices of its shard that it receives from the R ranks (one flat buffer
 * per source rank, padding zero), its fp32 master/m/v shard and its bf16
 * parameter shard; dpg_reduce_scatter_adam on the shard plan, with the R
 * received buffers in rank order as `grads`, then computes exactly the
 * values of shard r of the single-device step (the same rank-ordered fp32
 * sums, scale and Adam), and per-bucket norms of that shard alone.  The
 * exchange itself (slice q of a rank's bucket to rank q before, the bf16
 * shards to every rank after) is the caller's collective.  Host only.
 * Free with dpg_plan_destroy. */
int dpg_plan_shards(const dpg_plan_t* plan, dpg_plan_t** out);
void dpg_plan_destroy(dpg_plan_t* plan);
/* Sizes of a plan; any output pointer may be NULL. */
int dpg_plan_info(const dpg_plan_t* plan, int32_t* n_params, int32_t* n_buckets,
                  int64_t* total_padded, int32_t* R);
/* Bucket b: element offset in the flat buffer, padded size, shard size. */
int dpg_plan_bucket(const dpg_plan_t* plan, int32_t b, int64_t* offset,
                    int64_t* padded_numel, int64_t* shard_numel);
/* Parameter p (registration index): bucket and element offset in the flat
 * buffer of its slice, and its element count. */
int dpg_plan_param(const dpg_plan_t* plan, int32_t p, int32_t* bucket,
                   int64_t* offset, int64_t* numel);
/* Bulk copy of the maps into caller host arrays (n_params / n_buckets
 * entries; any pointer may be NULL). */
int dpg_plan_export(const dpg_plan_t* plan, int32_t* param_bucket, int64_t* param_offset,
                    int64_t* bucket_offset, int64_t* bucket_padded);
/* Upload the plan's tables to the current device (synchronous; idempotent). */
int dpg_plan_upload(dpg_plan_t* plan);

/* ---------------------------------------------------------------------------
 * Pack / unpack (one replica)       ["Parallelisms" -- FSDP / Flat parameter]
 * param_grads: HOST array of n_params DEVICE pointers to bf16 gradients
 * (2-byte aligned; NULL allowed only for zero-size parameters).
 * dpg_pack:   flat[offset_p + i] = grad_p[i]; every padding slot set to 0.
 * dpg_unpack: grad_p[i] = flat[offset_p + i]; padding is not read.
 * In steady state gradients are views into the flat buffer and no pack runs.
 * ------------------------------------------------------------------------- */
int dpg_pack(const dpg_plan_t* plan, const void* const* param_grads, void* flat_bf16,
             void* stream);
int dpg_unpack(const dpg_plan_t* plan, const void* flat_bf16, void* const* param_grads,
               void* stream);

/* ---------------------------------------------------------------------------
 * Checkpoint and resharding of the optimizer state  ["Distributed Training
 *      and Parallelism" -- Reproduction and debugging: checkpoint ownership,
 *      resumability, mesh reconfiguration]
 * The canonical layout is independent of the plan: parameters back to back
 * in REGISTRATION order, no padding, element j of parameter p at
 * sum(numels[0..p)) + j.  A state exported under one plan imports under any
 * plan of the same parameter list (another R or cap_bytes), which is how the
 * state moves to a different data-parallel layout.
 * flat[k] / canon[k], k < n_arrays (1..8): DEVICE pointers to fp32 arrays
 * (e.g. master, exp_avg, exp_avg_sq); flat arrays hold total_padded elements
 * (32-byte aligned), canonical arrays sum(numels) elements (4-byte aligned).
 * dpg_export_state: canon[k][c_p + j] = flat[k][offset_p + j].
 * dpg_import_state: flat[k][offset_p + j] = canon[k][c_p + j]; every padding
 * slot of flat[k] is set to 0.
 * The step counter t is the caller's (dpg_hparams.step) and travels with it.
 * ------------------------------------------------------------------------- */
#define DPG_MAX_STATE_ARRAYS 8
int dpg_export_state(const dpg_plan_t* plan, const float* const* flat, float* const* canon,
                     int32_t n_arrays, void* stream);
int dpg_import_state(const dpg_plan_t* plan, const float* const* canon, float* const* flat,
                     int32_t n_arrays, void* stream);

/* ---------------------------------------------------------------------------
 * no_sync gradient accumulation (one replica)   ["Distributed Training and
 *                    Parallelism" -- Data parallelism and the global gradient]
 * acc_f32[i] = f32(g[i]) if first != 0, else acc_f32[i] + f32(g[i]) (binary32,
 * round to nearest), for all total_padded elements.  The final microbatch is
 * not accumulated here: pass it as last_micro_bf16 to the reduction below.
 * ------------------------------------------------------------------------- */
int dpg_accumulate(const dpg_plan_t* plan, const void* flat_bf16, float* acc_f32,
                   int32_t first, void* stream);

/* ---------------------------------------------------------------------------
 * Paired no_sync accumulation (no counterpart on the pages: a schedule of the
 * same sums for a caller that keeps TWO bf16 gradient buffers per replica)
 * acc_f32[i] = f32(a[i]) + f32(b[i]) if first != 0, else
 * (acc_f32[i] + f32(a[i])) + f32(b[i]): exactly the two binary32 additions of
 * dpg_accumulate(a) then dpg_accumulate(b), in that order, with the fp32
 * buffer read and written once instead of twice (8 or 12 bytes per element
 * instead of 16 or 20).  micro_a is the earlier microbatch.
 * ------------------------------------------------------------------------- */
int dpg_accumulate_pair(const dpg_plan_t* plan, const void* micro_a_bf16,
                        const void* micro_b_bf16, float* acc_f32, int32_t first, void* stream);

/* ---------------------------------------------------------------------------
 * Whole step with the LAST TWO microbatches folded into the reduction (same
 * schedule note as dpg_accumulate_pair)
 * Replica r's contribution is x_r = (acc_f32[r] + f32(micro_a[r])) +
 * f32(micro_b[r]) -- what dpg_accumulate(micro_a) followed by dpg_step with
 * last_micro_bf16 = micro_b computes, bit for bit -- then the rank-ordered
 * sum, scale, Adam and cast exactly as dpg_step.  micro_a/micro_b: R
 * DEVICE (or page-locked host) bf16 flat buffers, 16-byte aligned;
 * acc_f32: R fp32 flat buffers, 32-byte aligned.  valid_tokens counts every
 * microbatch of the cycle (R*K counts).  Norm outputs as dpg_step.
 * ------------------------------------------------------------------------- */
/* ---------------------------------------------------------------------------
 * Deferred accumulation: the step of a K-microbatch cycle with no
 * accumulation pass before it
 *      ["Distributed Training and Parallelism" -- Data parallelism and the
 *       global gradient (no_sync: no intermediate reductions; the global
 *       count covers every microbatch)]
 * A caller that keeps each replica's K microbatch gradients in K bf16 flat
 * buffers (2K bytes per parameter per replica, against 4 + 2 for one fp32
 * accumulator and one bf16 buffer) hands them all to the fused pass, which
 * computes for every element
 *   x_r = ((f32(g[r][0]) + f32(g[r][1])) + ...) + f32(g[r][K-1])   (binary32)
 *   s   = x_0 + x_1 + ... + x_{R-1}                               (rank order)
 * -- exactly the sums of K-1 dpg_accumulate passes followed by dpg_step with
 * the last microbatch fused -- then scales, runs Adam and casts as dpg_step.
 * One pass moves 2KR + 26 bytes per parameter for the whole cycle.
 * micro_bf16: HOST array of R*K DEVICE (or page-locked host) pointers,
 *   replica-major (micro_bf16[r*K + k] = microbatch k of replica r), 16-byte
 *   aligned; 1 <= K and R*K <= DPG_MAX_REPLICAS (else DPG_ERR_INVALID_ARG).
 * valid_tokens counts every microbatch of the cycle (R*K counts).  Norm
 * outputs as dpg_step.  Always the chunked launch (a grid cap set with
 * dpg_set_fused_max_ctas does not apply).
 * ------------------------------------------------------------------------- */
int dpg_step_deferred(const dpg_plan_t* plan, const void* const* micro_bf16, int32_t K,
                      const int64_t* valid_tokens, int32_t n_counts, const dpg_hparams* hp,
                      float* master, float* exp_avg, float* exp_avg_sq, void* const* param_views,
                      int32_t n_views, float* bucket_sqnorm, int64_t* bucket_nonfinite,
                      void* stream);

int dpg_step_fold2(const dpg_plan_t* plan, const float* const* acc_f32,
                   const void* const* micro_a_bf16, const void* const* micro_b_bf16,
                   const int64_t* valid_tokens, int32_t n_counts, const dpg_hparams* hp,
                   float* master, float* exp_avg, float* exp_avg_sq, void* const* param_views,
                   int32_t n_views, float* bucket_sqnorm, int64_t* bucket_nonfinite,
                   void* stream);

/* ---------------------------------------------------------------------------
 * Fused reduce-scatter + normalisation + Adam + all-gather, buckets [b0, b1)
 *      ["Parallelisms" -- ZeRO-1, ZeRO-2; "Parallelism Starts With the
 *       Bottleneck" -- Allreduce equals reducescatter plus allgather;
 *       "Distributed Training and Parallelism" -- Data parallelism and the
 *       global gradient; Kingma & Ba Alg. 1]
 * For every element i of every shard of buckets b0..b1-1, in one pass:
 *   x_r = f32(grads[r][i])                         (grads_dtype == DPG_BF16)
 *       | grads[r][i]                              (DPG_F32: fp32 accumulation)
 *   x_r = x_r + f32(last_micro_bf16[r][i])         (if last_micro_bf16 != NULL)
 *   s   = x_0 + x_1 + ... + x_{R-1}                (binary32, rank order)
 *   g   = s * fp32(1/G),  G = sum(valid_tokens[0..n_counts))   (int64)
 *   Adam on master/exp_avg/exp_avg_sq (see dpg_hparams), binary32, no FMA
 *   param_views[k][i] = bf16_rne(master[i])        (k < n_views)
 * grads: HOST array of R device pointers to flat buffers (R = plan's R).
 * last_micro_bf16: NULL or HOST array of R device pointers (flat bf16).
 * valid_tokens: HOST array (e.g. R*K counts); each >= 0; G == 0 -> error.
 * master, exp_avg, exp_avg_sq: flat fp32, updated in place.
 * param_views: HOST array of n_views device pointers to flat bf16 buffers
 *   (0 <= n_views <= DPG_MAX_VIEWS; views alias one buffer in the usual case).
 * bucket_sqnorm (nullable, device, n_buckets floats): entry b receives the
 *   sum over bucket b of g*g (fp32 partials summed in double; deterministic).
 * bucket_nonfinite (nullable, device, n_buckets int64): count of elements of
 *   bucket b whose g is NaN or infinite (they are propagated, not skipped).
 * reduced_grad (nullable, device, flat fp32): receives g (debug/parity).
 * 0 <= b0 <= b1 <= n_buckets; b0 == b1 does nothing and returns DPG_OK.
 * The gradient buffers' padding slots must hold zeros (dpg_pack writes them).
 * ------------------------------------------------------------------------- */
int dpg_reduce_scatter_adam(const dpg_plan_t* plan, const void* const* grads,
                            int32_t grads_dtype, const void* const* last_micro_bf16,
                            const int64_t* valid_tokens, int32_t n_counts,
                            const dpg_hparams* hp, float* master, float* exp_avg,
                            float* exp_avg_sq, void* const* param_views, int32_t n_views,
                            float* bucket_sqnorm, int64_t* bucket_nonfinite,
                            float* reduced_grad, int32_t b0, int32_t b1, void* stream);

/* ---------------------------------------------------------------------------
 * The same update issued bucket by bucket as the backward pass finishes each
 *      ["Parallelisms" -- Gradient bucketing, Critical path: a bucket is
 *       reduced as soon as its gradients are ready, overlapping the rest of
 *       the backward]
 * For b = b0 .. b1-1 in order: `stream` waits on ready_events[b - b0] (a
 * cudaEvent_t the producer records once bucket b's gradients are complete in
 * every replica; HOST array of b1 - b0 handles), then bucket b's update is
 * launched on `stream` -- one fused launch (and, with a norm output, one
 * finalize) per bucket, issued from C++ without returning to the caller.
 * Arguments and results otherwise as dpg_reduce_scatter_adam over [b0, b1),
 * to the bit.  All arguments are checked before the stream is given any
 * wait or launch; a NULL ready_events (b1 > b0) or a NULL handle is
 * DPG_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------- */
int dpg_reduce_scatter_adam_when_ready(const dpg_plan_t* plan, const void* const* grads,
                                       int32_t grads_dtype, const void* const* last_micro_bf16,
                                       const int64_t* valid_tokens, int32_t n_counts,
                                       const dpg_hparams* hp, float* master, float* exp_avg,
                                       float* exp_avg_sq, void* const* param_views,
                                       int32_t n_views, float* bucket_sqnorm,
                                       int64_t* bucket_nonfinite, float* reduced_grad, int32_t b0,
                                       int32_t b1, void* const* ready_events, void* stream);

/* ---------------------------------------------------------------------------
 * All-gather / cast on its own, buckets [b0, b1)
 *      ["Parallelisms" -- ZeRO-1: workers all-gather the updated shards]
 * param_views[k][i] = bf16_rne(master[i]) for every element of the buckets.
 * ------------------------------------------------------------------------- */
int dpg_allgather_params(const dpg_plan_t* plan, const float* master,
                         void* const* param_views, int32_t n_views, int32_t b0, int32_t b1,
                         void* stream);

/* ---------------------------------------------------------------------------
 * ZeRO-3 parameter all-gather, buckets [b0, b1)   ["Parallelisms" -- ZeRO-3:
 *      before a layer runs in forward, and again in backward, workers
 *      all-gather its parameter shards; "Parallelism Strategies in
 *      Distributed Computing" -- ZeRO and FSDP]
 * param_bf16: the flat bf16 parameter buffer in which every rank's shard of
 * every bucket lives in place (shard r of bucket b at its shard range);
 * views[k][i] = param_bf16[i] for every element of the buckets: each
 * replica's full copy of the layer, assembled from all shards.  Under ZeRO-3
 * the step itself then writes only the sharded parameters (n_views = 1 on the
 * shared buffer), and layers are gathered before use.
 * ------------------------------------------------------------------------- */
int dpg_gather_params_bf16(const dpg_plan_t* plan, const void* param_bf16,
                           void* const* param_views, int32_t n_views, int32_t b0, int32_t b1,
                           void* stream);

/* ---------------------------------------------------------------------------
 * One whole optimizer step over every bucket (one fused launch plus, when a
 * norm output is requested, one small finalize launch).  Same arguments and
 * semantics as dpg_reduce_scatter_adam with b0 = 0, b1 = n_buckets and no
 * reduced-gradient output.
 * ------------------------------------------------------------------------- */
int dpg_step(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
             const void* const* last_micro_bf16, const int64_t* valid_tokens,
             int32_t n_counts, const dpg_hparams* hp, float* master, float* exp_avg,
             float* exp_avg_sq, void* const* param_views, int32_t n_views,
             float* bucket_sqnorm, int64_t* bucket_nonfinite, void* stream);

/* ---------------------------------------------------------------------------
 * DDP / FSDP NO_SHARD schedule, buckets [b0, b1)   ["Parallelisms" -- Data
 *      parallel; FSDP (NO_SHARD all-reduces gradients like DDP); "Parallelism
 *      Strategies in Distributed Computing" -- DP and DDP]
 * dpg_allreduce_grads: reduced_grad[i] = (x_0 + ... + x_{R-1}) * fp32(1/G)
 *   for every element (x_r as in dpg_reduce_scatter_adam; rank order,
 *   binary32): the all-reduce result that every DDP replica receives.
 *   reduced_grad: device, flat fp32 (32-byte aligned).  bucket_sqnorm /
 *   bucket_nonfinite (nullable) as in dpg_reduce_scatter_adam.
 * dpg_adam_from_reduced: one replica's optimizer step on its own full copy
 *   of master/exp_avg/exp_avg_sq from reduced_grad (Adam as in
 *   dpg_reduce_scatter_adam, bf16 views written).  Under DDP each of the R
 *   replicas calls it on its own state: R times the optimizer traffic of the
 *   ZeRO-2 step, with bit-identical results (the test suite checks it).
 * ------------------------------------------------------------------------- */
int dpg_allreduce_grads(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                        const void* const* last_micro_bf16, const int64_t* valid_tokens,
                        int32_t n_counts, float* reduced_grad, float* bucket_sqnorm,
                        int64_t* bucket_nonfinite, int32_t b0, int32_t b1, void* stream);
int dpg_adam_from_reduced(const dpg_plan_t* plan, const float* reduced_grad, const dpg_hparams* hp,
                          float* master, float* exp_avg, float* exp_avg_sq,
                          void* const* param_views, int32_t n_views, float* bucket_sqnorm,
                          int64_t* bucket_nonfinite, int32_t b0, int32_t b1, void* stream);

/* ---------------------------------------------------------------------------
 * One whole step with global gradient-norm clipping   ["Parallelisms" --
 *      ZeRO-2: clipping needs the norm over all gradient shards before any
 *      weight is updated; only the local squared norms are all-reduced]
 * Same arguments and semantics as dpg_step, except that the normalised
 * reduced gradient g of every element is first multiplied by
 *   coef = fp32( min(1, max_norm / (||g||_2 + 1e-6)) ),
 * ||g||_2 over ALL buckets (squares of the fp32 g summed exactly in double,
 * square root and quotient in double; a NaN norm gives a NaN coefficient).
 * Pass 1 reduces and scales every element and sums its squares per bucket;
 * the coefficient is computed on the device (no host synchronisation); pass
 * 2 applies g * coef to Adam and writes the bf16 view(s).
 * max_norm: finite, > 0.  bucket_sqnorm / bucket_nonfinite (nullable): of the
 * UNclipped g.  reduced_grad (nullable, device, flat fp32, 32-byte aligned):
 * when given, pass 1 stores g there and pass 2 reads it instead of reading
 * the R replicas again ((2R+34) instead of (4R+26) bytes per parameter).
 * clip_out (nullable, device float[2]): receives {||g||_2, coef}.
 * Uses the plan's scratch like dpg_step (same no-overlap rule).
 * ------------------------------------------------------------------------- */
int dpg_step_clipped(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                     const void* const* last_micro_bf16, const int64_t* valid_tokens,
                     int32_t n_counts, const dpg_hparams* hp, double max_norm, float* master,
                     float* exp_avg, float* exp_avg_sq, void* const* param_views, int32_t n_views,
                     float* bucket_sqnorm, int64_t* bucket_nonfinite, float* reduced_grad,
                     float* clip_out, void* stream);

/* ---------------------------------------------------------------------------
 * dpg_step through the STAGED variant of the fused pass: in each CTA a
 * producer warp copies the R gradient slices and the master/m/v slices of the
 * units it will process (half a 4096-element tile at R = 8, a whole tile at
 * R <= 4) into a ring of shared-memory stages with the
 * bulk-copy engine (cp.async.bulk, completion counted in bytes on a "full"
 * mbarrier per stage), refilling a stage as soon as the consumer warps have
 * released it on its "empty" mbarrier.  Same arguments and results as dpg_step for bf16 gradients
 * (grads_dtype must be DPG_BF16, no last microbatch), R in {1, 2, 4, 8}.
 * Every device-side wait is bounded (1 s); a wait that runs out makes the
 * CTA wait (bounded) for its own copies in flight and return, and records
 * DPG_ERR_DEVICE_TIMEOUT in the plan's status word: the outputs are then
 * incomplete.  dpg_check_device_status() synchronises `stream` and returns
 * that status (DPG_OK or DPG_ERR_DEVICE_TIMEOUT).
 * ------------------------------------------------------------------------- */
int dpg_step_staged(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                    const int64_t* valid_tokens, int32_t n_counts, const dpg_hparams* hp,
                    float* master, float* exp_avg, float* exp_avg_sq, void* const* param_views,
                    int32_t n_views, float* bucket_sqnorm, int64_t* bucket_nonfinite,
                    void* stream);
int dpg_check_device_status(const dpg_plan_t* plan, void* stream);

/* ---------------------------------------------------------------------------
 * dpg_step without any device allocation.  The pages have no counterpart to
 * this entry point: it exists for callers that must not have the library
 * allocate device memory -- for example code whose device memory is owned
 * by another allocator (a framework's caching pool or a fixed memory
 * budget), or that cannot accept the implicit synchronisation of
 * cudaMalloc/cudaFree in the middle of a training step.
 *
 * Same arguments, semantics and results as dpg_step (it runs the persistent
 * grid-stride form of the fused pass, so its per-bucket norms are summed in
 * another grouping, within their tolerance).  Instead of the plan's
 * device copy and norm scratch (which dpg_step allocates on first use), it
 * uses one static device array of DPG_NOALLOC_SCRATCH_BYTES compiled into the
 * library, which every GPU that loads the library holds until the process
 * exits.  That array holds the bucket tables (16 bytes per bucket, copied in
 * from the plan's host tables on `stream` at every call) and, when a norm
 * output is requested, the norm partials of the launch: 196 bytes for each
 * bucket visit of each CTA, where a CTA visits min(buckets, ceil(tiles / CTAs))
 * buckets at most (tiles of 4096 elements, one CTA per SM) -- about 2.5 MB for
 * a 1.2B-parameter model in 83 buckets on 152 SMs.  Each section is rounded
 * up to 256 bytes.  A plan whose launch does not fit is rejected with
 * DPG_ERR_INVALID_ARG before any device work.  Nothing in the array needs to
 * start at zero: each call rewrites the tables and every partial it reads.
 * The call never calls cudaMalloc, cudaFree or any allocating routine.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, once per device, with that device current); make
 * that first call before any stream capture.  Every call shares the one
 * array, so calls whose device work overlaps (for example on two streams)
 * race and must not be issued.
 * ------------------------------------------------------------------------- */
#define DPG_NOALLOC_SCRATCH_BYTES (8u << 20)
int dpg_step_noalloc(const dpg_plan_t* plan, const void* const* grads, int32_t grads_dtype,
                     const void* const* last_micro_bf16, const int64_t* valid_tokens,
                     int32_t n_counts, const dpg_hparams* hp, float* master, float* exp_avg,
                     float* exp_avg_sq, void* const* param_views, int32_t n_views,
                     float* bucket_sqnorm, int64_t* bucket_nonfinite, void* stream);

/* Launch shape -------------------------------------------------------------- */
/* By default the fused passes (dpg_step, dpg_reduce_scatter_adam,
 * dpg_step_fold2, dpg_adam_from_reduced, dpg_allreduce_grads and
 * dpg_step_clipped -- whose norm pass stays on the persistent grid when it
 * only re-reads R <= 4 replicas) launch one small CTA per 1024-element chunk,
 * which keeps
 * the most bytes in flight.  max_ctas > 0 makes later launches from the
 * CALLING THREAD use instead a persistent grid of at most max_ctas CTAs
 * (grid-stride over 4096-element tiles), leaving SMs free for work running
 * concurrently on other streams at the cost of the pass's own bandwidth;
 * dpg_step_noalloc always uses the persistent grid and honours the bound
 * too.  0 restores the default.
 * Results are the same bits for any launch shape; only the per-bucket norms'
 * summation grouping changes (within their documented tolerance).
 * Negative: DPG_ERR_INVALID_ARG. */
int dpg_set_fused_max_ctas(int32_t max_ctas);

/* Programmatic dependent launch (a Hopper / Blackwell stream feature).  With
 * on = 1 (the default) the chunked fused kernels, their norm finalize and
 * clip coefficient, and the accumulation, all-gather and gather kernels are
 * launched from the CALLING THREAD with programmatic stream serialization:
 * the GPU may schedule such a kernel while the previous kernel of the stream
 * is still draining, which shortens the gap between short back-to-back
 * launches (per-bucket updates, layer-by-layer gathers).  Each of these
 * kernels waits on the device, before its first memory access, until the
 * previous kernel has completed and its writes are visible, so stream order
 * and results are exactly those of plain launches.  on = 0 launches them
 * plainly.  Anything other than 0 or 1: DPG_ERR_INVALID_ARG. */
int dpg_set_programmatic_launch(int32_t on);

/* Diagnostics -------------------------------------------------------------- */
/* Number of kernels this library has launched since it was loaded. */
int64_t dpg_launch_count(void);
/* The next fused reduce-scatter-Adam launch issued by the calling thread
 * records start_event immediately before itself and stop_event immediately
 * after itself, on its own stream (cudaEvent_t handles created by the caller);
 * the request is then cleared.  NULL, NULL clears a pending request.  Lets a
 * caller time the fused kernel alone inside a whole step. */
int dpg_time_next_fused_launch(void* start_event, void* stop_event);
/* Index checks.  A library built with `python -m zero_optimizer_step_gb300.build
 * --debug` (libdpg_debug.so, compiled with DPG_DEBUG) checks, in the kernels
 * that derive indices from the plan's device tables -- the chunked fused and
 * norm passes, the chunk finalize, pack/unpack -- every element and table
 * index before using it.  A failed check skips its access and records the
 * first failure in a word of the plan; it never faults or traps.
 * dpg_debug_checks: *built = 1 for such a library, 0 otherwise;
 * *first_failure = the first failure recorded for `plan` since the last call
 * ((code << 32) | CTA index; codes 1 fused or norm pass, 2 finalize of a
 * long bucket, 3 finalize of a short bucket, 4 pack/unpack; 0 = none), which
 * it then clears.  Synchronizes the device in a checking build.  No
 * counterpart on the pages. */
int dpg_debug_checks(const dpg_plan_t* plan, int32_t* built, int64_t* first_failure);
/* Test hook of a checking build: index checks of later launches from the
 * calling thread bound element indices by `limit` instead of the plan's
 * total (limit < 0 restores it), so that a test can make a check fail
 * without any out-of-range access.  Honoured only by a checking build and
 * only when DPG_TEST_HOOKS is "1" in the environment; otherwise
 * DPG_ERR_INVALID_ARG. */
int dpg_debug_set_limit(int64_t limit);

/* Test-only fault injection for the staged step: its next launch by the
 * calling thread never fetches unit `skip_unit` (-1: none), so the CTA
 * that owns it must run out its wait, and every wait is bounded by
 * `timeout_ns` (<= 0: the default 1 s).  Used to test the timeout path.
 * Honoured only when the environment variable DPG_TEST_HOOKS is "1" at the
 * time of the call; otherwise it changes nothing and returns
 * DPG_ERR_INVALID_ARG. */
int dpg_set_staged_fault(int64_t skip_unit, int64_t timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* DPG_H */
