/*
 * fsdp_oracle.c -- plain CPU oracle for the FSDP FlatParameter step.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the bench's
 * CPU-baseline / reference leg load this file's library. It shares no code,
 * header, table or helper with the CUDA library and includes none of it.
 * It is deliberately slow and literal: one pass per step of the method,
 * element by element, in the order the sources state, so that it can be
 * checked against them by eye. The only concession to speed is an OpenMP
 * "parallel for" over independent elements, which changes no arithmetic.
 *
 * Sources (page title -- section):
 *  [ANN]   "Fully Sharded Data Parallel: faster AI training with fewer GPUs"
 *          (techreport.ngo) -- "From all-reduce to sharded parameters":
 *          all-reduce = reduce-scatter + all-gather, blocks summed per rank
 *          index (first figure caption); each GPU updates its local shard
 *          (second figure caption); FSDP gives results identical to DDP;
 *          "Harnessing FSDP's full power", item 3: a unit's parameters are
 *          flattened into one tensor with one set of hyperparameters.
 *  [GUIDE] "FSDP (Fully Sharded Data Parallel)" (vanos001.github.io) --
 *          "The Sharding Scheme": P/N params, P/N grads, 4P/N fp32 Adam
 *          state (m, v, master) per worker; "The Per-Layer Communication":
 *          all-gather before forward and backward, reduce-scatter after
 *          backward; "Mixed Precision and FSDP": bf16 compute copy, fp32
 *          master and optimizer state.
 *  [FAIR]  "fairseq ... Fully Sharded Data Parallel (FSDP) 实战指南"
 *          (zskr.cn) -- "参数定义与底层实现": --fp32-reduce-scatter reduces the
 *          gradients in FP32, compute_dtype is fp16 under --fp16;
 *          "限制与兼容性说明": FSDP is exact for pointwise optimizers (Adam,
 *          AdamW, ...) and relies on parameter flattening; "与 PyTorch DDP
 *          的对比": training results identical to DDP.
 *  [DP]    "Data Parallelism" (vanos001.github.io) -- "The Basic Protocol":
 *          G_avg = (1/N) sum_i G_i, then W = W - lr * Adam(G_avg, m, v).
 *
 * Precision. The sources fix fp32 for the reduce-scatter accumulation ([FAIR]
 * --fp32-reduce-scatter) and for the master weights and Adam state ([GUIDE]),
 * so the oracle's step runs in fp32, one IEEE-rounded operation at a time
 * (built with -ffp-contract=off: no fused multiply-add). An fp64 shadow
 * (orc_*_f64) restates the same definitions in double to bound that rounding.
 *
 * Readings where the sources are silent (readings of them, not statements in them):
 *  R1 padding: zeros appended at the end up to ceil(P/N)*N; no gaps between
 *     parameters.
 *  R2 reduction order: fp32, ranks 0..N-1, starting from G_0.
 *  R3 average and loss-scale unscale: one multiply by c = 1/(N*scale), c
 *     computed in double and rounded once to float.
 *  R4 AdamW: decoupled weight decay applied to the weight before the Adam
 *     update; bias-corrected moments; eps added outside the square root.
 *     Host scalars (computed in double, rounded once to float):
 *     decay = 1 - lr*wd, 1-beta1, 1-beta2, alpha = lr/(1-beta1^t),
 *     b2s = sqrt(1-beta2^t). Per element, in this order:
 *        p = p*decay; m = beta1*m + (1-beta1)*g; v = beta2*v + (1-beta2)*(g*g);
 *        denom = sqrt(v)/b2s + eps; p = p - alpha*(m/denom).
 *  R5 weight decay applies to every element (one parameter group per unit).
 *  R6 cast: IEEE round-to-nearest-even; overflow to infinity; NaN stays a
 *     (quiet) NaN.
 *  R7 m = v = 0 before step 1; t counts from 1.
 *  R17-R19 the SGD-momentum, Adamax and Adadelta rules of orc_step_ex.
 *  R20 a reduce-scatter in the gradient dtype rounds every partial sum.
 *  R21 low-precision state: widen, update in fp32, round each value back.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F16 2

/* ------------------------------------------------------------------ */
/* threads                                                              */
/* ------------------------------------------------------------------ */

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* layout: flatten, pad, shard, views            [ANN] item 3, R1      */
/* ------------------------------------------------------------------ */

/* ceil(numel / world) * world, the FlatParameter length after padding (R1).
 * Returns -1 for numel < 0 or world < 1. */
int64_t orc_padded_numel(int64_t numel, int64_t world) {
    if (numel < 0 || world < 1) return -1;
    int64_t shards = numel / world;
    if (shards * world < numel) shards += 1;
    return shards * world;
}

/* Each rank owns an equal block of the padded FlatParameter ([ANN] first
 * figure caption, [GUIDE] "The Sharding Scheme"): S = P_pad / N. */
int64_t orc_shard_numel(int64_t padded, int64_t world) {
    if (padded < 0 || world < 1 || padded % world != 0) return -1;
    return padded / world;
}

/* Offsets of the original parameters inside the FlatParameter: the
 * parameters are concatenated in registration order ([ANN] item 3). */
void orc_view_offsets(const int64_t *numels, int n, int64_t *offsets) {
    int64_t at = 0;
    for (int k = 0; k < n; ++k) {
        offsets[k] = at;
        at += numels[k];
    }
}

/* Concatenate n tensors of elem_size-byte elements into dst and zero the
 * padding [sum(numels), padded). */
void orc_flatten_pad(const void *const *srcs, const int64_t *numels, int n,
                     int elem_size, int64_t padded, void *dst) {
    unsigned char *out = (unsigned char *)dst;
    int64_t at = 0;
    for (int k = 0; k < n; ++k) {
        memcpy(out + at * elem_size, srcs[k], (size_t)(numels[k] * elem_size));
        at += numels[k];
    }
    if (padded > at) memset(out + at * elem_size, 0, (size_t)((padded - at) * elem_size));
}

/* ------------------------------------------------------------------ */
/* number formats                                              R6       */
/* ------------------------------------------------------------------ */

static uint32_t f32_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    return u;
}

static float bits_f32(uint32_t u) {
    float x;
    memcpy(&x, &u, 4);
    return x;
}

/* bfloat16 keeps the top 16 bits of the binary32 pattern. Round to nearest,
 * ties to even: drop the low 16 bits, add one unit when the dropped part is
 * above one half, or exactly one half with an odd kept part. A carry out of
 * the mantissa moves into the exponent, which is the correctly rounded
 * result (up to infinity). */
uint16_t orc_f32_to_bf16(float x) {
    uint32_t u = f32_bits(x);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN: keep sign and payload top, set quiet bit */
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
    return (uint16_t)kept;
}

float orc_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. Written from the
 * format: the value is |x| = M * 2^(e-23) with M the 24-bit significand. */
uint16_t orc_f32_to_f16(float x) {
    uint32_t u = f32_bits(x);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t ef = (u >> 23) & 0xffu;
    uint32_t frac = u & 0x007fffffu;
    if (ef == 0xffu) {
        if (frac) return (uint16_t)(sign | 0x7e00u | (frac >> 13)); /* quiet NaN */
        return (uint16_t)(sign | 0x7c00u);                          /* infinity */
    }
    if (ef == 0) return sign; /* binary32 zero or subnormal: below half of the smallest binary16 subnormal */
    int e = (int)ef - 127;
    uint64_t M = (uint64_t)frac | 0x00800000u;
    if (e > 15) return (uint16_t)(sign | 0x7c00u); /* |x| >= 2^16: overflow */
    if (e >= -14) {
        /* normal range: keep 11 significant bits, drop 13 */
        uint32_t kept = (uint32_t)(M >> 13);           /* 1xxxxxxxxxx (11 bits) */
        uint32_t dropped = (uint32_t)(M & 0x1fffu);
        uint32_t h = ((uint32_t)(e + 15) << 10) | (kept & 0x3ffu);
        if (dropped > 0x1000u || (dropped == 0x1000u && (kept & 1u))) h += 1u; /* may carry to the next binade / infinity */
        return (uint16_t)(sign | h);
    }
    /* subnormal range: value in units of 2^-24 is M * 2^(e+1); shift right by -(e+1) */
    int shift = -(e + 1); /* >= 14 */
    if (shift > 40) return sign;
    uint64_t kept = M >> shift;
    uint64_t dropped = M & (((uint64_t)1 << shift) - 1);
    uint64_t half = (uint64_t)1 << (shift - 1);
    if (dropped > half || (dropped == half && (kept & 1u))) kept += 1; /* may become the smallest normal 0x0400 */
    return (uint16_t)(sign | (uint16_t)kept);
}

float orc_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t ef = (h >> 10) & 0x1fu;
    uint32_t frac = h & 0x3ffu;
    if (ef == 0x1fu) return bits_f32(sign | 0x7f800000u | (frac << 13));
    if (ef == 0) {
        /* subnormal: frac * 2^-24, exact in binary32 */
        float mag = (float)frac * 5.9604644775390625e-8f; /* 2^-24 */
        return sign ? -mag : mag;
    }
    return bits_f32(sign | ((ef + 112u) << 23) | (frac << 13));
}

void orc_cast_array(const float *x, int64_t n, int dtype, uint16_t *out) {
    if (dtype == ORC_BF16) {
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(x[i]);
    } else {
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(x[i]);
    }
}

void orc_cast_bits_array(const uint32_t *bits, int64_t n, int dtype, uint16_t *out) {
    orc_cast_array((const float *)bits, n, dtype, out);
}

void orc_widen_array(const uint16_t *h, int64_t n, int dtype, float *out) {
    if (dtype == ORC_BF16) {
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f32(h[i]);
    } else {
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f32(h[i]);
    }
}

static float grad_at(const void *base, int dtype, int64_t j) {
    if (dtype == ORC_F32) return ((const float *)base)[j];
    uint16_t h = ((const uint16_t *)base)[j];
    return dtype == ORC_BF16 ? orc_bf16_to_f32(h) : orc_f16_to_f32(h);
}

static int dtype_size(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

/* ------------------------------------------------------------------ */
/* hyperparameters -> per-step scalars                      R3, R4, R7  */
/* ------------------------------------------------------------------ */

typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int64_t step;      /* t >= 1 */
    float grad_scale;  /* static loss scale; 1 when there is none */
} orc_hparams;

typedef struct {
    float c;              /* 1/(N*scale) */
    float decay;          /* 1 - lr*wd */
    float beta1, beta2;
    float one_minus_beta1, one_minus_beta2;
    float alpha;          /* lr / (1 - beta1^t) */
    float b2s;            /* sqrt(1 - beta2^t) */
    float eps;
} orc_scalars;

int orc_scalars_from_hparams(const orc_hparams *h, int64_t world, orc_scalars *s) {
    if (!h || !s || world < 1 || h->step < 1 || !(h->grad_scale > 0.0f)) return 1;
    double t = (double)h->step;
    s->c = (float)(1.0 / ((double)world * (double)h->grad_scale));
    s->decay = (float)(1.0 - (double)h->lr * (double)h->weight_decay);
    s->beta1 = h->beta1;
    s->beta2 = h->beta2;
    s->one_minus_beta1 = (float)(1.0 - (double)h->beta1);
    s->one_minus_beta2 = (float)(1.0 - (double)h->beta2);
    s->alpha = (float)((double)h->lr / (1.0 - pow((double)h->beta1, t)));
    s->b2s = (float)sqrt(1.0 - pow((double)h->beta2, t));
    s->eps = h->eps;
    return 0;
}

/* ------------------------------------------------------------------ */
/* the step, one source step per function                              */
/* ------------------------------------------------------------------ */

/* Reduce-scatter, [ANN] first figure caption + [DP] "The Basic Protocol":
 * rank `rank` receives block `rank` of the sum of the N ranks' gradients,
 * averaged: g[i] = (sum_q G_q[rank*S + i]) * c, in fp32 ([FAIR]
 * --fp32-reduce-scatter), q in rank order (R2). */
void orc_reduce_scatter(const void *const *G, int grad_dtype, int64_t N, int64_t S,
                        int64_t rank, float c, float *g) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < S; ++i) {
        int64_t j = rank * S + i;
        float acc = grad_at(G[0], grad_dtype, j);
        for (int64_t q = 1; q < N; ++q) acc = acc + grad_at(G[q], grad_dtype, j);
        g[i] = acc * c;
    }
}

/* The DDP all-reduce average over the whole flat buffer, [DP] "The Basic
 * Protocol" step 3: G_avg[j] = (sum_q G_q[j]) * c for every j. */
void orc_all_reduce_avg(const void *const *G, int grad_dtype, int64_t N, int64_t P_pad,
                        float c, float *G_avg) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < P_pad; ++j) {
        float acc = grad_at(G[0], grad_dtype, j);
        for (int64_t q = 1; q < N; ++q) acc = acc + grad_at(G[q], grad_dtype, j);
        G_avg[j] = acc * c;
    }
}

/* Pointwise AdamW on n elements ([FAIR] "限制与兼容性说明": the optimizer is
 * pointwise, so it runs on the local shard alone; [DP] step 4; R4, R5). */
void orc_adamw(float *p, float *m, float *v, const float *g, int64_t n, const orc_scalars *s) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float gi = g[i];
        float pi = p[i] * s->decay;
        float mi = s->beta1 * m[i] + s->one_minus_beta1 * gi;
        float vi = s->beta2 * v[i] + s->one_minus_beta2 * (gi * gi);
        float denom = sqrtf(vi) / s->b2s + s->eps;
        pi = pi - s->alpha * (mi / denom);
        p[i] = pi;
        m[i] = mi;
        v[i] = vi;
    }
}

/* Cast of the fp32 master shard to the compute dtype ([GUIDE] "Mixed
 * Precision and FSDP"; [FAIR] compute_dtype), R6. ORC_F32 copies. */
void orc_cast(const float *p, int64_t n, int out_dtype, void *out) {
    if (out_dtype == ORC_F32) {
        memcpy(out, p, (size_t)n * 4);
        return;
    }
    orc_cast_array(p, n, out_dtype, (uint16_t *)out);
}

/* All-gather, [ANN] first figure caption + [GUIDE] "The Per-Layer
 * Communication": every rank receives all N shards, block r from rank r:
 * full[r*S + i] = shard_r[i]. */
void orc_all_gather(const void *const *shards, int elem_size, int64_t N, int64_t S, void *full) {
    unsigned char *out = (unsigned char *)full;
    for (int64_t r = 0; r < N; ++r)
        memcpy(out + (size_t)(r * S) * elem_size, shards[r], (size_t)S * elem_size);
}

/* One FSDP step of one unit with N ranks emulated one after another
 * ([ANN] second figure caption; [GUIDE] "The Per-Layer Communication"):
 *   for each rank r: reduce-scatter block r -> g; AdamW on rank r's shard of
 *   master/m/v (stored at offset r*S of the concatenated buffers); cast into
 *   rank r's own shard buffer shards_out + r*S;
 *   then all-gather the N shards into out_full.
 * g_scratch holds S floats. Returns nonzero on bad arguments. */
int orc_fsdp_step(const void *const *G, int grad_dtype, int64_t N, int64_t P_pad,
                  float *master, float *m, float *v, int out_dtype, void *shards_out,
                  void *out_full, const orc_hparams *h, float *g_scratch) {
    orc_scalars s;
    int64_t S = orc_shard_numel(P_pad, N);
    if (S < 0 || orc_scalars_from_hparams(h, N, &s)) return 1;
    int es = dtype_size(out_dtype);
    const void *shard_ptrs[4096];
    if (N > 4096) return 1;
    for (int64_t r = 0; r < N; ++r) {
        orc_reduce_scatter(G, grad_dtype, N, S, r, s.c, g_scratch);
        orc_adamw(master + r * S, m + r * S, v + r * S, g_scratch, S, &s);
        unsigned char *shard_r = (unsigned char *)shards_out + (size_t)(r * S) * es;
        orc_cast(master + r * S, S, out_dtype, shard_r);
        shard_ptrs[r] = shard_r;
    }
    orc_all_gather(shard_ptrs, es, N, S, out_full);
    return 0;
}

/* The DDP reference of the same step ([DP] "The Basic Protocol"): all-reduce
 * average over the whole buffer, a full-replica AdamW, a full cast. The
 * sources state FSDP's results are identical to this ([ANN]; [FAIR] "与
 * PyTorch DDP 的对比"). g_scratch holds P_pad floats. */
int orc_ddp_step(const void *const *G, int grad_dtype, int64_t N, int64_t P_pad,
                 float *master, float *m, float *v, int out_dtype, void *out_full,
                 const orc_hparams *h, float *g_scratch) {
    orc_scalars s;
    if (P_pad < 0 || orc_scalars_from_hparams(h, N, &s)) return 1;
    orc_all_reduce_avg(G, grad_dtype, N, P_pad, s.c, g_scratch);
    orc_adamw(master, m, v, g_scratch, P_pad, &s);
    orc_cast(master, P_pad, out_dtype, out_full);
    return 0;
}

/* ------------------------------------------------------------------ */
/* variants of the step: other optimizers, reduce and state precisions */
/* ------------------------------------------------------------------ */

/* Optimizers. [FAIR] "限制与兼容性说明": FSDP is compatible with the
 * pointwise optimizers (Adam, AdamW, Adadelta, Adamax, SGD, ...); [ANN]
 * "Where FSDP goes next": tested with SGD and Adam. The pages print none of
 * the update rules; these are the textbook rules (readings R17-R19):
 *  SGD with momentum mu (no dampening), L2 weight decay added to the gradient:
 *     d = g + wd*p;  b = d on the first step, else b = mu*b + d;  p = p - lr*b
 *  Adamax (Kingma & Ba, the infinity-norm variant of Adam), L2 decay:
 *     d = g + wd*p;  m = b1*m + (1-b1)*d;  u = max(b2*u, |d| + eps) (NaN if
 *     either side is NaN);  p = p - alpha * (m/u), alpha = lr/(1-b1^t) as
 *     for AdamW
 *  Adadelta (Zeiler), lr multiplier, L2 decay, rho = beta1:
 *     d = g + wd*p;  s = rho*s + (1-rho)*(d*d);
 *     delta = (sqrt(a + eps) / sqrt(s + eps)) * d;  a = rho*a + (1-rho)*(delta*delta);
 *     p = p - lr*delta */
#define ORC_OPT_ADAMW 0
#define ORC_OPT_SGD 1
#define ORC_OPT_ADAMAX 2
#define ORC_OPT_ADADELTA 3

static int opt_states(int opt) { return opt == ORC_OPT_SGD ? 1 : 2; }

/* One element of one optimizer, fp32, one rounding per operation. */
static void update_elem(int opt, float g, float *p, float *s0, float *s1, const orc_scalars *s,
                        const orc_hparams *h) {
    float pi = *p;
    if (opt == ORC_OPT_ADAMW) {
        float mi = *s0, vi = *s1;
        pi = pi * s->decay;
        mi = s->beta1 * mi + s->one_minus_beta1 * g;
        vi = s->beta2 * vi + s->one_minus_beta2 * (g * g);
        float denom = sqrtf(vi) / s->b2s + s->eps;
        pi = pi - s->alpha * (mi / denom);
        *s0 = mi;
        *s1 = vi;
    } else if (opt == ORC_OPT_SGD) {
        float d = g + h->weight_decay * pi;
        float b = h->step == 1 ? d : h->beta1 * *s0 + d;
        pi = pi - h->lr * b;
        *s0 = b;
    } else if (opt == ORC_OPT_ADAMAX) {
        float d = g + h->weight_decay * pi;
        float mi = s->beta1 * *s0 + s->one_minus_beta1 * d;
        float a = s->beta2 * *s1, b = fabsf(d) + s->eps;
        float ui = (a > b || a != a) ? a : b; /* max, NaN if either side is NaN */
        pi = pi - s->alpha * (mi / ui);
        *s0 = mi;
        *s1 = ui;
    } else { /* ORC_OPT_ADADELTA */
        float d = g + h->weight_decay * pi;
        float sq = s->beta1 * *s0 + s->one_minus_beta1 * (d * d);
        float delta = (sqrtf(*s1 + s->eps) / sqrtf(sq + s->eps)) * d;
        float acc = s->beta1 * *s1 + s->one_minus_beta1 * (delta * delta);
        pi = pi - h->lr * delta;
        *s0 = sq;
        *s1 = acc;
    }
    *p = pi;
}

static float load_as_f32(const void *base, int dtype, int64_t j) { return grad_at(base, dtype, j); }

static void store_from_f32(void *base, int dtype, int64_t j, float x) {
    if (dtype == ORC_F32)
        ((float *)base)[j] = x;
    else if (dtype == ORC_BF16)
        ((uint16_t *)base)[j] = orc_f32_to_bf16(x);
    else
        ((uint16_t *)base)[j] = orc_f32_to_f16(x);
}

static float round_to(int dtype, float x) {
    if (dtype == ORC_BF16) return orc_bf16_to_f32(orc_f32_to_bf16(x));
    if (dtype == ORC_F16) return orc_f16_to_f32(orc_f32_to_f16(x));
    return x;
}

/* Reduce-scatter summed in the gradient dtype: the default without
 * --fp32-reduce-scatter ([FAIR] "参数定义与底层实现"), and the "FP16
 * reduce-scatter on gradients" of [ANN] "Harnessing FSDP's full power" item 4.
 * Reading R20: ranks in order, each partial sum computed in fp32 and rounded
 * to the gradient dtype; then g = acc * c in fp32. */
void orc_reduce_scatter_lowp(const void *const *G, int grad_dtype, int64_t N, int64_t S, int64_t rank, float c,
                             float *g) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < S; ++i) {
        int64_t j = rank * S + i;
        float acc = grad_at(G[0], grad_dtype, j);
        for (int64_t q = 1; q < N; ++q) acc = round_to(grad_dtype, acc + grad_at(G[q], grad_dtype, j));
        g[i] = acc * c;
    }
}

/* The step with a chosen optimizer, reduce precision and state precision,
 * all N ranks emulated in turn, then the all-gather ([GUIDE] "The Per-Layer
 * Communication").
 *  state_dtype ORC_F32: `param` is the fp32 master; the shard written to
 *     shards_out is its cast to out_dtype.
 *  state_dtype ORC_BF16 / ORC_F16 ([GUIDE] "Mixed Precision and FSDP":
 *     without fp32 master, params and Adam state in bf16; [ANN] item 4: FP16
 *     master weights): `param` and the states are stored in that dtype, each
 *     element widened to fp32, updated as above, rounded back (R21); the
 *     param itself is the shard (out_dtype must equal state_dtype).
 * s1 may be NULL for SGD. g_scratch holds S floats. Returns nonzero on bad
 * arguments. */
int orc_step_ex(int opt, int reduce_lowp, const void *const *G, int grad_dtype, int64_t N, int64_t P_pad,
                void *param, void *s0, void *s1, int state_dtype, int out_dtype, void *shards_out,
                void *out_full, const orc_hparams *h, float *g_scratch) {
    orc_scalars sc;
    int64_t S = orc_shard_numel(P_pad, N);
    if (S < 0 || orc_scalars_from_hparams(h, N, &sc) || opt < 0 || opt > 3) return 1;
    if (state_dtype != ORC_F32 && out_dtype != state_dtype) return 1;
    if (opt_states(opt) == 2 && !s1) return 1;
    int es = dtype_size(out_dtype);
    const void *shard_ptrs[4096];
    if (N > 4096) return 1;
    for (int64_t r = 0; r < N; ++r) {
        if (reduce_lowp)
            orc_reduce_scatter_lowp(G, grad_dtype, N, S, r, sc.c, g_scratch);
        else
            orc_reduce_scatter(G, grad_dtype, N, S, r, sc.c, g_scratch);
        unsigned char *shard_r = (unsigned char *)shards_out + (size_t)(r * S) * es;
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < S; ++i) {
            int64_t j = r * S + i;
            float p = load_as_f32(param, state_dtype, j);
            float a = load_as_f32(s0, state_dtype, j);
            float b = s1 ? load_as_f32(s1, state_dtype, j) : 0.0f;
            update_elem(opt, g_scratch[i], &p, &a, &b, &sc, h);
            store_from_f32(param, state_dtype, j, p);
            store_from_f32(s0, state_dtype, j, a);
            if (s1) store_from_f32(s1, state_dtype, j, b);
            store_from_f32(shard_r, out_dtype, i, p);
        }
        shard_ptrs[r] = shard_r;
    }
    orc_all_gather(shard_ptrs, es, N, S, out_full);
    return 0;
}

/* ------------------------------------------------------------------ */
/* fp64 shadow: the same definitions in double                          */
/* ------------------------------------------------------------------ */

/* G_avg = (1/(N*scale)) * sum_q G_q, in double. */
void orc_all_reduce_avg_f64(const void *const *G, int grad_dtype, int64_t N, int64_t P_pad,
                            double grad_scale, double *G_avg) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < P_pad; ++j) {
        double acc = 0.0;
        for (int64_t q = 0; q < N; ++q) acc += (double)grad_at(G[q], grad_dtype, j);
        G_avg[j] = acc / ((double)N * grad_scale);
    }
}

/* AdamW with decoupled weight decay in its textbook form, in double:
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   mhat = m/(1-b1^t);    vhat = v/(1-b2^t);
 *   p = p - lr*wd*p - lr*mhat/(sqrt(vhat) + eps). */
void orc_adamw_f64(double *p, double *m, double *v, const double *g, int64_t n,
                   const orc_hparams *h) {
    double b1 = h->beta1, b2 = h->beta2, lr = h->lr, wd = h->weight_decay, eps = h->eps;
    double t = (double)h->step;
    double bc1 = 1.0 - pow(b1, t), bc2 = 1.0 - pow(b2, t);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double gi = g[i];
        m[i] = b1 * m[i] + (1.0 - b1) * gi;
        v[i] = b2 * v[i] + (1.0 - b2) * gi * gi;
        double mhat = m[i] / bc1, vhat = v[i] / bc2;
        p[i] = p[i] - lr * wd * p[i] - lr * mhat / (sqrt(vhat) + eps);
    }
}
