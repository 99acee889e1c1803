/*
 * oracle.c -- plain, single-threaded CPU oracle for the data-parallel ZeRO-2
 * gradient step (bucket plan, pack/unpack, no_sync accumulation, fixed-order
 * reduce-scatter, token normalisation, mixed-precision Adam, bf16 all-gather).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file; only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC -lm
 * (-ffp-contract=off matters: aarch64 GCC would otherwise fuse a*b+c into one
 * FMA and change the rounding of every step below.)
 *
 * Every floating-point operation is an IEEE-754 binary32 operation with
 * round-to-nearest-even, written one operation per statement so that the
 * order of rounding is the order on the page.  Constants that depend only on
 * the hyper-parameters are computed once in binary64 and rounded once to
 * binary32.
 *
 * Sources (web pages; section names as printed on them):
 *  [P1] "Parallelisms" (vladislavkruglikov.com): sections "Data parallel",
 *       "Gradient bucketing", "ZeRO-1", "ZeRO-2", "FSDP" / "Flat parameter".
 *  [P2] "Distributed Training and Parallelism" (naatyu.github.io atlas):
 *       sections "Data parallelism and the global gradient", "ZeRO and
 *       sharded state", "Infer communication from matrix layouts".
 *  [P3] "Parallelism Strategies in Distributed Computing" (voidindex):
 *       "Comparison / Cost per strategy", "DP and DDP", "ZeRO and FSDP".
 *  [P4] "Parallelism Starts With the Bottleneck" (rajdeepmondal.com):
 *       "Allreduce equals reducescatter plus allgather", "Data parallelism is
 *       simple and pays for it in memory", "ZeRO removes the copies".
 *  [KB] Kingma & Ba, "Adam: A Method for Stochastic Optimization" (ICLR 2015),
 *       Algorithm 1.  The pages name Adam and its state but print no formula.
 *
 * Every function is pinned by a test against something other than itself
 * (page-printed numbers, closed forms, invariants, library routines, brute
 * force); no function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_EZERO_TOKENS -2

#define ORACLE_BF16 0
#define ORACLE_F32 1

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                              */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static float bits_f32(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* bf16 -> fp32 is exact: a bf16 value is the upper half of a binary32. */
float oracle_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* fp32 -> bf16, round to nearest, ties to even (IEEE-754 default rounding).
 * The kept part is the upper 16 bits; the dropped part is the lower 16 bits,
 * compared against one half of the kept part's last place (0x8000).  A carry
 * out of the significand moves into the exponent, which is the correct
 * result (the largest finite values round up to infinity).  A NaN keeps its
 * sign and leading payload bits and is made quiet. */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u = f32_bits(f);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u) {
        return (uint16_t)(kept | 0x0040u); /* NaN -> quiet NaN */
    }
    if (dropped > 0x8000u) {
        kept += 1u;
    } else if (dropped == 0x8000u) {
        if (kept & 1u) kept += 1u; /* tie: round to the even neighbour */
    }
    return (uint16_t)kept;
}

void oracle_f32_to_bf16_array(const float* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f32_to_bf16(x[i]);
}

void oracle_bf16_to_f32_array(const uint16_t* x, float* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_bf16_to_f32(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Bucket plan  [P1 "Data parallel", "Gradient bucketing", "Flat parameter";  */
/*               P2 "Data parallelism and the global gradient"]               */
/* ------------------------------------------------------------------------ */
/*
 * Gradients of later layers are ready first in backward, so parameters are
 * registered into buckets in REVERSE order of their registration.  A bucket
 * is one flat buffer; each parameter's gradient is a view into a slice of it.
 *
 * Rules (readings where the pages are silent):
 *  - a parameter's slice starts at the next multiple of 8 elements (16 bytes);
 *  - a bucket's size is its end offset in elements times 2 bytes (bf16
 *    gradients); a parameter with elements that would push a bucket that
 *    already holds elements over cap_bytes closes that bucket first; a
 *    parameter larger than the cap therefore sits alone; parameters are never
 *    split; a zero-size parameter never closes a bucket;
 *  - a closed bucket is padded with zeros to a multiple of 8*R elements, so
 *    that it splits into R equal shards of whole 8-element vectors; shard r
 *    of bucket b is [r*N_b/R, (r+1)*N_b/R) inside the bucket [P1 "ZeRO-2"];
 *  - buckets are laid out one after another in the flat buffer, in the order
 *    they are closed (bucket 0 holds the last-registered parameters).
 *
 * Outputs (caller allocates n entries for the per-param arrays and n entries
 * for the per-bucket arrays; at most n buckets exist):
 *   param_bucket[p], param_offset[p] (element offset in the whole flat buffer)
 *   bucket_offset[b], bucket_padded[b], *n_buckets, *total_padded.
 */
int oracle_plan_buckets(const int64_t* numels, int32_t n, int64_t cap_bytes,
                        int32_t R, int32_t* param_bucket, int64_t* param_offset,
                        int64_t* bucket_offset, int64_t* bucket_padded,
                        int32_t* n_buckets, int64_t* total_padded) {
    if (n < 0 || cap_bytes <= 0 || R < 1) return ORACLE_EINVAL;
    for (int32_t p = 0; p < n; ++p)
        if (numels[p] < 0) return ORACLE_EINVAL;

    int32_t nb = 0;          /* buckets closed so far */
    int64_t flat_base = 0;   /* offset of the open bucket in the flat buffer */
    int64_t used = 0;        /* elements used in the open bucket */
    int32_t members = 0;     /* parameters placed in the open bucket */
    int64_t* local = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!local) return ORACLE_EINVAL;

    for (int32_t p = n - 1; p >= 0; --p) {
        int64_t start = (used + 7) / 8 * 8;
        int64_t end = start + numels[p];
        if (used > 0 && numels[p] > 0 && end * 2 > cap_bytes) {
            /* close the open bucket */
            int64_t unit = 8 * (int64_t)R;
            int64_t padded = (used + unit - 1) / unit * unit;
            bucket_offset[nb] = flat_base;
            bucket_padded[nb] = padded;
            flat_base += padded;
            nb += 1;
            used = 0;
            members = 0;
            start = 0;
            end = numels[p];
        }
        param_bucket[p] = nb;
        local[p] = start;
        used = end;
        members += 1;
    }
    if (members > 0) {
        int64_t unit = 8 * (int64_t)R;
        int64_t padded = (used + unit - 1) / unit * unit;
        bucket_offset[nb] = flat_base;
        bucket_padded[nb] = padded;
        flat_base += padded;
        nb += 1;
    }
    for (int32_t p = 0; p < n; ++p)
        param_offset[p] = bucket_offset[param_bucket[p]] + local[p];
    free(local);
    *n_buckets = nb;
    *total_padded = flat_base;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Pack / unpack  [P1 "Flat parameter": originals become views into slices]  */
/* ------------------------------------------------------------------------ */

/* flat[param_offset[p] + i] = grads[p][i]; every other slot is zero. */
void oracle_pack(int32_t n, const int64_t* numels, const int64_t* param_offset,
                 const uint16_t* const* grads, int64_t total, uint16_t* flat) {
    for (int64_t i = 0; i < total; ++i) flat[i] = 0;
    for (int32_t p = 0; p < n; ++p)
        for (int64_t i = 0; i < numels[p]; ++i) flat[param_offset[p] + i] = grads[p][i];
}

/* grads[p][i] = flat[param_offset[p] + i]. */
void oracle_unpack(int32_t n, const int64_t* numels, const int64_t* param_offset,
                   const uint16_t* flat, uint16_t* const* grads) {
    for (int32_t p = 0; p < n; ++p)
        for (int64_t i = 0; i < numels[p]; ++i) grads[p][i] = flat[param_offset[p] + i];
}

/* ------------------------------------------------------------------------ */
/* Checkpoint layout  [P2 "Reproduction and debugging": checkpoint            */
/* ownership, resumability, mesh reconfiguration]                            */
/* ------------------------------------------------------------------------ */
/*
 * The canonical layout of a state array holds the parameters back to back in
 * registration order with no padding; it does not depend on the bucket plan.
 */
void oracle_export_state(int32_t n, const int64_t* numels, const int64_t* param_offset,
                         const float* flat, float* canon) {
    int64_t c = 0;
    for (int32_t p = 0; p < n; ++p) {
        for (int64_t i = 0; i < numels[p]; ++i) canon[c + i] = flat[param_offset[p] + i];
        c += numels[p];
    }
}

/* flat = 0 everywhere, then every parameter's slice from the canonical array. */
void oracle_import_state(int32_t n, const int64_t* numels, const int64_t* param_offset,
                         const float* canon, int64_t total, float* flat) {
    for (int64_t i = 0; i < total; ++i) flat[i] = 0.0f;
    int64_t c = 0;
    for (int32_t p = 0; p < n; ++p) {
        for (int64_t i = 0; i < numels[p]; ++i) flat[param_offset[p] + i] = canon[c + i];
        c += numels[p];
    }
}

/* ------------------------------------------------------------------------ */
/* Gradient accumulation without synchronisation  [P2 "Data parallelism and */
/* the global gradient": no_sync on intermediate microbatches]               */
/* ------------------------------------------------------------------------ */

/* first != 0: acc = fp32(g);  otherwise acc = acc + fp32(g). */
void oracle_accumulate(int64_t n, const uint16_t* g, float* acc, int32_t first) {
    for (int64_t i = 0; i < n; ++i) {
        float x = oracle_bf16_to_f32(g[i]);
        if (first) {
            acc[i] = x;
        } else {
            float s = acc[i] + x;
            acc[i] = s;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Token normalisation  [P2 "Data parallelism and the global gradient"]      */
/* ------------------------------------------------------------------------ */
/*
 * Each rank's gradient is that of its local SUMMED loss.  Scaling a local
 * summed loss by R/G and then averaging over the R ranks gives
 * (1/R) * sum_r (R/G) g_r = sum_r g_r / G, the gradient of the global mean
 * loss over G valid tokens.  The combined factor 1/G is applied once, as one
 * binary32 multiply by fp32(1/G) after the rank-ordered sum.  G counts every
 * rank and every accumulated microbatch.  G == 0 is an error.
 */
int oracle_grad_scale(const int64_t* tokens, int32_t n_counts, float* scale) {
    if (n_counts < 1) return ORACLE_EINVAL;
    int64_t G = 0;
    for (int32_t i = 0; i < n_counts; ++i) {
        if (tokens[i] < 0) return ORACLE_EINVAL;
        G += tokens[i];
    }
    if (G == 0) return ORACLE_EZERO_TOKENS;
    double inv = 1.0 / (double)G;
    *scale = (float)inv;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Reduction across replicas  [P1 "ZeRO-1"/"ZeRO-2"; P4 "Allreduce equals   */
/* reducescatter plus allgather"]                                             */
/* ------------------------------------------------------------------------ */

static float replica_value(const void* const* grads, int32_t dtype,
                           const uint16_t* const* last, int32_t r, int64_t i) {
    float x;
    if (dtype == ORACLE_BF16) {
        x = oracle_bf16_to_f32(((const uint16_t*)grads[r])[i]);
    } else {
        x = ((const float*)grads[r])[i];
    }
    if (last) {
        /* the final microbatch is added to the fp32 accumulation here */
        float y = oracle_bf16_to_f32(last[r][i]);
        x = x + y;
    }
    return x;
}

/*
 * out[i] = (x_0[i] + x_1[i] + ... + x_{R-1}[i]) * scale, summed in rank order
 * 0..R-1 in binary32 starting from x_0 (not from 0.0, which would turn -0
 * into +0), then multiplied once by scale.  Elements [lo, hi) of the buffers.
 */
void oracle_reduce_range(int32_t R, const void* const* grads, int32_t dtype,
                         const uint16_t* const* last, float scale, int64_t lo,
                         int64_t hi, float* out) {
    for (int64_t i = lo; i < hi; ++i) {
        float s = replica_value(grads, dtype, last, 0, i);
        for (int32_t r = 1; r < R; ++r) {
            float x = replica_value(grads, dtype, last, r, i);
            s = s + x;
        }
        float g = s * scale;
        out[i] = g;
    }
}

/* All-reduce without sharding: every rank receives the full reduced buffer.
 * out_per_rank[r] is rank r's copy.  Used only to check RS o AG == AR. */
void oracle_allreduce(int32_t R, int64_t n, const void* const* grads, int32_t dtype,
                      const uint16_t* const* last, float scale, float* const* out_per_rank) {
    for (int32_t dst = 0; dst < R; ++dst)
        oracle_reduce_range(R, grads, dtype, last, scale, 0, n, out_per_rank[dst]);
}

/* ------------------------------------------------------------------------ */
/* Global gradient-norm clipping  [P1 "ZeRO-2": the norm over all gradient    */
/* shards is needed before any weight is updated]                             */
/* ------------------------------------------------------------------------ */
/*
 * ||g||_2 over every element of the normalised reduced gradient (squares of
 * the binary32 values summed in binary64 in index order), and the clip
 * coefficient min(1, max_norm / (||g|| + 1e-6)) computed in binary64 and
 * rounded once to binary32 (the convention of torch.nn.utils.clip_grad_norm_;
 * a NaN norm gives a NaN coefficient).
 */
void oracle_clip_coef(const float* g, int64_t n, double max_norm, double* norm_out,
                      float* coef_out) {
    double total = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double x = (double)g[i];
        total += x * x;
    }
    double norm = sqrt(total);
    double c = max_norm / (norm + 1e-6);
    if (c > 1.0) c = 1.0;
    *norm_out = norm;
    *coef_out = (float)c;
}

/* g[i] = g[i] * coef (binary32). */
void oracle_scale_range(float* g, int64_t n, float coef) {
    for (int64_t i = 0; i < n; ++i) {
        float y = g[i] * coef;
        g[i] = y;
    }
}

/* ------------------------------------------------------------------------ */
/* Mixed-precision Adam on one shard  [P1 "ZeRO-1": m, v, step counter and   */
/* fp32 master weight; KB Algorithm 1]                                        */
/* ------------------------------------------------------------------------ */

typedef struct {
    float beta1, beta2, one_minus_beta1, one_minus_beta2;
    float bias1, bias2, lr, eps, lr_wd;
    int decay;
} adam_consts;

static int adam_setup(double lr, double beta1, double beta2, double eps, double wd,
                      int64_t t, adam_consts* c) {
    if (t < 1) return ORACLE_EINVAL;
    if (!(beta1 >= 0.0 && beta1 < 1.0 && beta2 >= 0.0 && beta2 < 1.0)) return ORACLE_EINVAL;
    c->beta1 = (float)beta1;
    c->beta2 = (float)beta2;
    c->one_minus_beta1 = (float)(1.0 - beta1);
    c->one_minus_beta2 = (float)(1.0 - beta2);
    c->bias1 = (float)(1.0 - pow(beta1, (double)t));
    c->bias2 = (float)(1.0 - pow(beta2, (double)t));
    c->lr = (float)lr;
    c->eps = (float)eps;
    c->lr_wd = (float)(lr * wd);
    c->decay = (wd != 0.0);
    return ORACLE_OK;
}

/*
 * For i in [lo, hi), with g[i] the normalised reduced gradient and t the step
 * number of this update (first update: t = 1):
 *   [decoupled weight decay, only when wd != 0: w <- w - (lr*wd) * w]
 *   m  <- beta1*m + (1-beta1)*g
 *   v  <- beta2*v + (1-beta2)*(g*g)
 *   mh <- m / (1-beta1^t)
 *   vh <- v / (1-beta2^t)
 *   w  <- w - lr * ( mh / (sqrt(vh) + eps) )
 */
int oracle_adam_range(const float* g, float* master, float* m, float* v, int64_t lo,
                      int64_t hi, double lr, double beta1, double beta2, double eps,
                      double wd, int64_t t) {
    adam_consts c;
    int st = adam_setup(lr, beta1, beta2, eps, wd, t, &c);
    if (st != ORACLE_OK) return st;
    for (int64_t i = lo; i < hi; ++i) {
        float gi = g[i];
        float w = master[i];
        if (c.decay) {
            float d = c.lr_wd * w;
            w = w - d;
        }
        float m_old = c.beta1 * m[i];
        float m_new_term = c.one_minus_beta1 * gi;
        float mi = m_old + m_new_term;
        float g2 = gi * gi;
        float v_old = c.beta2 * v[i];
        float v_new_term = c.one_minus_beta2 * g2;
        float vi = v_old + v_new_term;
        float m_hat = mi / c.bias1;
        float v_hat = vi / c.bias2;
        float root = sqrtf(v_hat);
        float denom = root + c.eps;
        float u = m_hat / denom;
        float step = c.lr * u;
        w = w - step;
        m[i] = mi;
        v[i] = vi;
        master[i] = w;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* The whole step  [P1 "ZeRO-1"/"ZeRO-2"; P4 "ZeRO removes the copies"]       */
/* ------------------------------------------------------------------------ */
/*
 * For every bucket b and every shard owner r (reduce-scatter):
 *   reduce the shard over the R replicas in rank order, scale by fp32(1/G),
 *   run Adam on the owner's slice of master/m/v.
 * Then the per-bucket sum of squared reduced gradients (the local squared
 * norm that a global clip would all-reduce, P1 "ZeRO-2"), in binary64.
 * Then the all-gather: every replica view receives bf16(master) for every
 * shard of every bucket.
 *
 * grads[r]: replica r's flat gradient buffer (bf16 or fp32 accumulation);
 * last[r]: replica r's final-microbatch bf16 buffer, or NULL.
 * views[k]: k-th bf16 parameter buffer to write (n_views may be 0).
 * reduced (nullable): receives the normalised reduced gradient.
 * sqnorm (nullable): per-bucket sum of g*g in binary64.
 */
int oracle_step(int32_t n_buckets, const int64_t* bucket_offset,
                const int64_t* bucket_padded, int32_t R, const void* const* grads,
                int32_t dtype, const uint16_t* const* last, const int64_t* tokens,
                int32_t n_counts, double lr, double beta1, double beta2, double eps,
                double wd, int64_t t, float* master, float* m, float* v,
                uint16_t* const* views, int32_t n_views, float* reduced, double* sqnorm) {
    float scale;
    int st = oracle_grad_scale(tokens, n_counts, &scale);
    if (st != ORACLE_OK) return st;
    adam_consts probe;
    st = adam_setup(lr, beta1, beta2, eps, wd, t, &probe);
    if (st != ORACLE_OK) return st;
    if (R < 1 || (dtype != ORACLE_BF16 && dtype != ORACLE_F32)) return ORACLE_EINVAL;

    int64_t total = 0;
    for (int32_t b = 0; b < n_buckets; ++b) {
        if (bucket_padded[b] % R != 0) return ORACLE_EINVAL;
        int64_t e = bucket_offset[b] + bucket_padded[b];
        if (e > total) total = e;
    }
    float* g = (float*)malloc(sizeof(float) * (size_t)(total > 0 ? total : 1));
    if (!g) return ORACLE_EINVAL;

    for (int32_t b = 0; b < n_buckets; ++b) {
        int64_t shard = bucket_padded[b] / R;
        for (int32_t owner = 0; owner < R; ++owner) {
            int64_t lo = bucket_offset[b] + owner * shard;
            int64_t hi = lo + shard;
            oracle_reduce_range(R, grads, dtype, last, scale, lo, hi, g);
            oracle_adam_range(g, master, m, v, lo, hi, lr, beta1, beta2, eps, wd, t);
        }
        if (sqnorm) {
            double acc = 0.0;
            for (int64_t i = bucket_offset[b]; i < bucket_offset[b] + bucket_padded[b]; ++i) {
                double gi = (double)g[i];
                acc += gi * gi;
            }
            sqnorm[b] = acc;
        }
    }
    for (int32_t k = 0; k < n_views; ++k)
        for (int32_t b = 0; b < n_buckets; ++b)
            for (int64_t i = bucket_offset[b]; i < bucket_offset[b] + bucket_padded[b]; ++i)
                views[k][i] = oracle_f32_to_bf16(master[i]);
    if (reduced)
        for (int64_t i = 0; i < total; ++i) reduced[i] = g[i];
    free(g);
    return ORACLE_OK;
}

/* bf16 all-gather on its own: views[k][i] = bf16(master[i]) for i < n. */
void oracle_allgather(int64_t n, const float* master, uint16_t* const* views, int32_t n_views) {
    for (int32_t k = 0; k < n_views; ++k)
        for (int64_t i = 0; i < n; ++i) views[k][i] = oracle_f32_to_bf16(master[i]);
}

/* ------------------------------------------------------------------------ */
/* Model-state memory per replica  [P3 "Comparison / Cost per strategy",     */
/* "DP and DDP", "ZeRO and FSDP"; P4 "Data parallelism is simple and pays    */
/* for it in memory"]                                                         */
/* ------------------------------------------------------------------------ */
/*
 * Bytes of persistent model state per replica for psi parameters on N ranks:
 * bf16 parameter 2, bf16 gradient 2, fp32 master + m + v 12.
 *   stage 0 (DDP):    (2 + 2 + 12) psi
 *   stage 1 (ZeRO-1): (2 + 2) psi + 12 psi / N
 *   stage 2 (ZeRO-2): 2 psi + (2 + 12) psi / N
 *   stage 3 (ZeRO-3): (2 + 2 + 12) psi / N
 * Temporary buckets, activations and allocator overhead are not counted.
 */
double oracle_model_state_bytes(int32_t stage, double psi, int32_t N) {
    const double param = 2.0, grad = 2.0, optim = 4.0 + 4.0 + 4.0;
    double n = (double)N;
    switch (stage) {
        case 0: return (param + grad + optim) * psi;
        case 1: return (param + grad) * psi + optim * psi / n;
        case 2: return param * psi + (grad + optim) * psi / n;
        case 3: return (param + grad + optim) * psi / n;
        default: return -1.0;
    }
}
