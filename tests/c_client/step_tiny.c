/*
 * A C client of the library: no Python, no PyTorch.  It plans the tiny
 * three-parameter case ([64,32], [32], [32,10], R = 4, 2048-byte buckets),
 * allocates every buffer with the CUDA runtime, runs one dpg_step, a second
 * step through dpg_reduce_scatter_adam_when_ready gated on per-bucket events
 * recorded on another stream, and one dpg_allgather_params, and compares
 * every output bit for bit with the oracle (a test-only C library) run on the
 * same inputs.  It also checks the layout of the plan's shard plan (the split
 * across R GPUs).
 * Exit status 0 on a match; prints the first mismatch otherwise.
 * Inputs: a fixed xorshift stream of normals (Box-Muller), plain and
 * reproducible; nothing here computes the method's arithmetic.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "dpg.h"

/* oracle (test infrastructure) */
int oracle_plan_buckets(const int64_t* numels, int32_t n, int64_t cap_bytes, int32_t R,
                        int32_t* param_bucket, int64_t* param_offset, int64_t* bucket_offset,
                        int64_t* bucket_padded, int32_t* n_buckets, int64_t* total_padded);
int oracle_step(int32_t n_buckets, const int64_t* bucket_offset, const int64_t* bucket_padded,
                int32_t R, const void* const* grads, int32_t dtype, const uint16_t* const* last,
                const int64_t* tokens, int32_t n_counts, double lr, double beta1, double beta2,
                double eps, double wd, int64_t t, float* master, float* m, float* v,
                uint16_t* const* views, int32_t n_views, float* reduced, double* sqnorm);
uint16_t oracle_f32_to_bf16(float f);

#define R 4
#define CHECK_CUDA(x)                                                                  \
    do {                                                                               \
        cudaError_t e_ = (x);                                                          \
        if (e_ != cudaSuccess) {                                                       \
            fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
            return 2;                                                                  \
        }                                                                              \
    } while (0)
#define CHECK_DPG(x)                                                                   \
    do {                                                                               \
        int s_ = (x);                                                                  \
        if (s_ != DPG_OK) {                                                            \
            fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, dpg_status_string(s_), \
                    dpg_last_error());                                                 \
            return 3;                                                                  \
        }                                                                              \
    } while (0)

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static double uniform01(void) {
    rng_state ^= rng_state << 13;
    rng_state ^= rng_state >> 7;
    rng_state ^= rng_state << 17;
    return ((rng_state >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}
static double normal(void) {
    const double u = uniform01(), w = uniform01();
    return sqrt(-2.0 * log(u)) * cos(6.283185307179586 * w);
}

static int same_bits(const void* a, const void* b, size_t bytes, const char* what) {
    if (memcmp(a, b, bytes) == 0) return 1;
    const unsigned char* x = (const unsigned char*)a;
    const unsigned char* y = (const unsigned char*)b;
    size_t i = 0;
    while (x[i] == y[i]) ++i;
    fprintf(stderr, "%s differs first at byte %zu\n", what, i);
    return 0;
}

int main(void) {
    if (dpg_abi_version() != DPG_ABI_VERSION) {
        fprintf(stderr, "ABI version mismatch\n");
        return 4;
    }
    const int64_t numels[3] = {64 * 32, 32, 32 * 10};
    const int64_t cap = 2048;
    dpg_plan_t* plan = NULL;
    CHECK_DPG(dpg_plan_buckets(numels, 3, cap, R, &plan));
    int32_t n_params = 0, n_buckets = 0, rr = 0;
    int64_t total = 0;
    CHECK_DPG(dpg_plan_info(plan, &n_params, &n_buckets, &total, &rr));

    /* the oracle's plan of the same list must be the library's */
    int32_t pb[3], onb = 0;
    int64_t po[3], bo[8], bp[8], ototal = 0;
    if (oracle_plan_buckets(numels, 3, cap, R, pb, po, bo, bp, &onb, &ototal) != 0 ||
        onb != n_buckets || ototal != total) {
        fprintf(stderr, "plan differs from the oracle's\n");
        return 5;
    }
    for (int32_t b = 0; b < n_buckets; ++b) {
        int64_t off = 0, pad = 0, shard = 0;
        CHECK_DPG(dpg_plan_bucket(plan, b, &off, &pad, &shard));
        if (off != bo[b] || pad != bp[b] || shard * R != pad) {
            fprintf(stderr, "bucket %d differs\n", b);
            return 5;
        }
    }

    /* the shard plan of the split across R GPUs: one bucket per bucket of
     * the plan, holding that bucket's shard, padded to a multiple of 8R */
    dpg_plan_t* shards = NULL;
    CHECK_DPG(dpg_plan_shards(plan, &shards));
    int32_t s_buckets = 0, s_r = 0;
    int64_t s_total = 0, s_expect = 0;
    CHECK_DPG(dpg_plan_info(shards, NULL, &s_buckets, &s_total, &s_r));
    if (s_buckets != n_buckets || s_r != R) {
        fprintf(stderr, "shard plan shape differs\n");
        return 6;
    }
    for (int32_t b = 0; b < n_buckets; ++b) {
        int64_t off = 0, pad = 0, soff = 0, spad = 0;
        CHECK_DPG(dpg_plan_bucket(plan, b, &off, &pad, NULL));
        CHECK_DPG(dpg_plan_bucket(shards, b, &soff, &spad, NULL));
        const int64_t want = (pad / R + 8 * R - 1) / (8 * R) * (8 * R);
        if (soff != s_expect || spad != want) {
            fprintf(stderr, "shard bucket %d differs\n", b);
            return 6;
        }
        s_expect += want;
    }
    if (s_total != s_expect) {
        fprintf(stderr, "shard plan size differs\n");
        return 6;
    }
    dpg_plan_destroy(shards);

    const size_t n = (size_t)total;
    uint16_t* hg[R];
    float* hw = (float*)malloc(n * sizeof(float));
    for (int r = 0; r < R; ++r) {
        hg[r] = (uint16_t*)calloc(n, sizeof(uint16_t));
        for (int p = 0; p < 3; ++p)     /* padding stays zero */
            for (int64_t j = 0; j < numels[p]; ++j)
                hg[r][po[p] + j] = oracle_f32_to_bf16((float)(normal() * 1e-2));
    }
    for (size_t i = 0; i < n; ++i) hw[i] = (float)(normal() * 0.02);
    const int64_t tokens[R] = {100, 80, 120, 60};

    /* device buffers owned by this program */
    void* dg[R];
    float *dw, *dm, *dv, *dsq;
    void *dview, *dview2;
    int64_t* dnf;
    for (int r = 0; r < R; ++r) {
        CHECK_CUDA(cudaMalloc(&dg[r], n * 2));
        CHECK_CUDA(cudaMemcpy(dg[r], hg[r], n * 2, cudaMemcpyHostToDevice));
    }
    CHECK_CUDA(cudaMalloc((void**)&dw, n * 4));
    CHECK_CUDA(cudaMalloc((void**)&dm, n * 4));
    CHECK_CUDA(cudaMalloc((void**)&dv, n * 4));
    CHECK_CUDA(cudaMalloc(&dview, n * 2));
    CHECK_CUDA(cudaMalloc(&dview2, n * 2));
    CHECK_CUDA(cudaMalloc((void**)&dsq, (size_t)n_buckets * 4));
    CHECK_CUDA(cudaMalloc((void**)&dnf, (size_t)n_buckets * 8));
    CHECK_CUDA(cudaMemcpy(dw, hw, n * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemset(dm, 0, n * 4));
    CHECK_CUDA(cudaMemset(dv, 0, n * 4));
    cudaStream_t s;
    CHECK_CUDA(cudaStreamCreate(&s));

    float* ow = (float*)malloc(n * 4);
    float* om = (float*)calloc(n, 4);
    float* ov = (float*)calloc(n, 4);
    uint16_t* oview = (uint16_t*)malloc(n * 2);
    double osq[8];
    memcpy(ow, hw, n * 4);
    const void* gptr[R];
    for (int r = 0; r < R; ++r) gptr[r] = hg[r];
    void* views[1] = {dview};
    /* the second step waits, bucket by bucket, on events a producer stream records */
    cudaStream_t producer;
    CHECK_CUDA(cudaStreamCreateWithFlags(&producer, cudaStreamNonBlocking));
    cudaEvent_t ready[8];
    if (n_buckets > 8) {
        fprintf(stderr, "unexpected bucket count %d\n", n_buckets);
        return 7;
    }
    for (int32_t b = 0; b < n_buckets; ++b) {
        CHECK_CUDA(cudaEventCreateWithFlags(&ready[b], cudaEventDisableTiming));
        CHECK_CUDA(cudaEventRecord(ready[b], producer));
    }
    for (int64_t t = 1; t <= 2; ++t) {
        dpg_hparams hp = {1e-3, 0.9, 0.999, 1e-8, 0.0, t};
        if (t == 1)
            CHECK_DPG(dpg_step(plan, (const void* const*)dg, DPG_BF16, NULL, tokens, R, &hp, dw,
                               dm, dv, views, 1, dsq, dnf, s));
        else
            CHECK_DPG(dpg_reduce_scatter_adam_when_ready(
                plan, (const void* const*)dg, DPG_BF16, NULL, tokens, R, &hp, dw, dm, dv, views,
                1, dsq, dnf, NULL, 0, n_buckets, (void* const*)ready, s));
        uint16_t* ov_ptr[1] = {oview};
        if (oracle_step(n_buckets, bo, bp, R, gptr, 0, NULL, tokens, R, 1e-3, 0.9, 0.999, 1e-8,
                        0.0, t, ow, om, ov, ov_ptr, 1, NULL, osq) != 0) {
            fprintf(stderr, "oracle_step failed\n");
            return 6;
        }
    }
    void* views2[1] = {dview2};
    CHECK_DPG(dpg_allgather_params(plan, dw, views2, 1, 0, n_buckets, s));
    CHECK_CUDA(cudaStreamSynchronize(s));

    float* gw = (float*)malloc(n * 4);
    float* gm = (float*)malloc(n * 4);
    float* gv = (float*)malloc(n * 4);
    uint16_t* gview = (uint16_t*)malloc(n * 2);
    uint16_t* gview2 = (uint16_t*)malloc(n * 2);
    CHECK_CUDA(cudaMemcpy(gw, dw, n * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(gm, dm, n * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(gv, dv, n * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(gview, dview, n * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(gview2, dview2, n * 2, cudaMemcpyDeviceToHost));
    int ok = same_bits(gw, ow, n * 4, "master") & same_bits(gm, om, n * 4, "exp_avg") &
             same_bits(gv, ov, n * 4, "exp_avg_sq") & same_bits(gview, oview, n * 2, "view") &
             same_bits(gview2, oview, n * 2, "all-gathered view");
    float gsq[8];
    CHECK_CUDA(cudaMemcpy(gsq, dsq, (size_t)n_buckets * 4, cudaMemcpyDeviceToHost));
    for (int32_t b = 0; b < n_buckets; ++b)
        if (fabs((double)gsq[b] - osq[b]) > 1e-5 * osq[b]) {
            fprintf(stderr, "bucket %d norm %.9g vs %.9g\n", b, gsq[b], osq[b]);
            ok = 0;
        }

    /* a G = 0 step is refused before any launch and writes nothing */
    const int64_t zeros[R] = {0, 0, 0, 0};
    dpg_hparams hp3 = {1e-3, 0.9, 0.999, 1e-8, 0.0, 3};
    if (dpg_step(plan, (const void* const*)dg, DPG_BF16, NULL, zeros, R, &hp3, dw, dm, dv, views,
                 1, dsq, dnf, s) != DPG_ERR_ZERO_TOKENS) {
        fprintf(stderr, "G = 0 not refused\n");
        ok = 0;
    }

    for (int r = 0; r < R; ++r) {
        cudaFree(dg[r]);
        free(hg[r]);
    }
    cudaFree(dw);
    cudaFree(dm);
    cudaFree(dv);
    cudaFree(dview);
    cudaFree(dview2);
    cudaFree(dsq);
    cudaFree(dnf);
    for (int32_t b = 0; b < n_buckets; ++b) cudaEventDestroy(ready[b]);
    cudaStreamDestroy(producer);
    cudaStreamDestroy(s);
    dpg_plan_destroy(plan);
    free(hw); free(ow); free(om); free(ov); free(oview);
    free(gw); free(gm); free(gv); free(gview); free(gview2);
    if (!ok) return 1;
    printf("C client: %lld elements, %d buckets, two steps (one event-gated) and an "
           "all-gather bit-exact\n",
           (long long)n, n_buckets);
    return 0;
}
