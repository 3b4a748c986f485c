/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the ZeRO-partitioned
 * mixed-precision Adam shard step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the tests, the smoke check of the package entry point and the
 * CPU-baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA library; the two meet only through seeded inputs.
 *
 * Every function writes out the plain definition of what the pages describe,
 * in the order they give it, with no blocking, fusion or reordering:
 *
 *   oracle_state_bytes   model-state bytes per device for stages 0-3
 *                        ("DeepSpeed ZeRO Stages" sec. 1.2 and 3.1-3.3;
 *                         "DeepSpeed ZeRO: Extreme Memory Efficiency",
 *                         "Three stages of partitioning the redundancy away")
 *   oracle_layout        flat-buffer partition into N_d disjoint shards
 *                        ("DeepSpeed ZeRO Stages" sec. 2, partition definition;
 *                         sec. 3.2, contiguous flat gradient buffer)
 *   oracle_grad_reduce   simulated reduce-scatter: N_d fp16 contributions,
 *                        summed, averaged and unscaled, plus the non-finite test
 *                        ("ZeRO Stage 1 Math", "The per-step mechanics", beat 2)
 *   oracle_adam_apply    elementwise Adam / AdamW on fp32 master, m, v and the
 *                        cast of the shard to fp16
 *                        ("DeepSpeed ZeRO Stages" sec. 2.1 Fact 1;
 *                         "ZeRO Stage 1 Math", "Where the 12 bytes come from"
 *                         and "The per-step mechanics", beat 3)
 *   oracle_shard_step    the two above for one shard with the skip rule
 *   oracle_commit        skip / commit bookkeeping after an overflow test
 *   oracle_grad_sqnorm,  global gradient-norm clipping: the squared norm of
 *   oracle_clip_factor,  the reduced gradient, the clip factor and the
 *   oracle_scale         scaled gradient ("DeepSpeed ZeRO Stages" sec. 2.1,
 *                        Fact 1: clipping needs ||g||_2 over all of P)
 *   oracle_sgd_apply     mixed-precision SGD with momentum on the shard, the
 *                        other optimizer the state multiplier K names
 *                        ("DeepSpeed ZeRO Stages" sec. 1.2)
 *   oracle_qwz_quantize, block-wise int8 quantization of the fp16 shard for
 *   oracle_qwz_dequantize the parameter all-gather and its inverse
 *                        ("ZeRO Optimization: Stages 1, 2, and 3 Explained",
 *                         ZeRO++ quantized weights; "DeepSpeed ZeRO Stages"
 *                         sec. 5.3, qwZ)
 *   oracle_adam8_maps,   8-bit Adam, the optimizer of K = 6 ("DeepSpeed ZeRO
 *   oracle_adam8_apply   Stages" sec. 1.2): m and v kept as 8-bit codes of a
 *                        dynamic map with a scale per block of 2048, after
 *                        Dettmers et al., "8-bit Optimizers via Block-wise
 *                        Quantization"
 *
 * Precision.  The pages fix the precisions: fp16 gradients and parameters,
 * fp32 master weights, m and v ("ZeRO Stage 1 Math", "The 16-bytes-per-
 * parameter budget").  So the update is evaluated in fp32, one IEEE
 * round-to-nearest operation per arithmetic step, and this file must be built
 * with -ffp-contract=off so that no multiply-add is fused.  Scalar
 * coefficients are formed in double and rounded once to float.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - bias correction m_hat = m / (1 - beta1^t), v_hat = v / (1 - beta2^t),
 *     t = number of applied updates including this one; beta^t is formed by
 *     t repeated double multiplications (no libm pow);
 *   - epsilon is added outside the square root, as printed;
 *   - weight decay is decoupled (AdamW): theta -= lr * (u + wd * theta);
 *   - the reduced gradient is sum_k fp32(h_k) in rank order 0..N_d-1, then one
 *     multiply by (float)(1 / (N_d * L)) for loss scale L;
 *   - overflow: any non-finite reduced gradient in the valid range skips the
 *     whole step; the loss scale halves, never below 1; no growth;
 *   - fp32 -> fp16 rounding is IEEE round-to-nearest-even;
 *   - clipping (the pages name it, give no formula): ||g||_2 over every
 *     shard of the reduced, unscaled gradient, summed in double;
 *     c = min(1, max_norm / (||g||_2 + 1e-6)) in double, rounded once to
 *     float, and g' = g * c in fp32 before the Adam update;
 *   - SGD with momentum (named with its K, no formula): the textbook rule,
 *     d = g + wd theta, b' = mu b + d (b = 0 before the first step),
 *     theta' = theta - lr b', fp32 master and fp32 momentum;
 *   - quantized weights (the pages give blocks with their own scale, 16 -> 8
 *     bit, nothing more): blocks of 256 consecutive parameters of the shard,
 *     the last one possibly shorter; scale = max|x| / 127 in fp32;
 *     q = rint(x / scale) (ties to even) in fp32, 0 when the scale is 0;
 *     the receiver rebuilds fp16(q * scale).
 *   - 8-bit Adam (named with its K, nothing more): block-wise quantization of
 *     m and v after Dettmers et al. (blocks of 2048, absmax scale, nearest
 *     code of a decimal-exponent map, signed for m and unsigned for v, ties
 *     to the smaller magnitude), fp32 master; the map's fraction values are
 *     the upper ends of their steps so that x = 1 is exact; the state is
 *     normalized as the method states it, state / absmax, one IEEE fp32
 *     division per element;
 *
 * Parity pins for every function live in the tests (closed forms and worked
 * values printed on the pages, exhaustive fp16 checks against numpy, the
 * textbook Adam of torch.optim in float64, hand-traced dyadic steps, brute-force
 * owner maps and the sharded == unsharded invariant).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32, written from the format definition.           */
/* ------------------------------------------------------------------------ */

/* Decode one binary16 value: 1 sign bit, 5 exponent bits (bias 15), 10
 * fraction bits.  Exact: every binary16 value is a binary32 value.  (The fp16
 * gradients and parameters of "ZeRO Stage 1 Math", "The 16-bytes-per-parameter
 * budget".) */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    float mag;
    if (expo == 0) {
        mag = ldexpf((float)frac, -24);               /* zero or subnormal */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexpf((float)(1024 + frac), expo - 25); /* (1.f) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

/* Round one binary32 value to binary16, ties to even (the fp16 cast of "ZeRO
 * Stage 1 Math", "The per-step mechanics", beat 3). */
uint16_t oracle_f32_to_f16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    double a = fabs((double)x);
    if (isinf(x) || a >= 65520.0)      /* 65520 is the midpoint of 65504 and 2^16 */
        return (uint16_t)(sign | 0x7c00);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                      /* a = f * 2^e, 0.5 <= f < 1 */
    int unbiased = e - 1;              /* a in [2^unbiased, 2^(unbiased+1)) */
    if (unbiased < -14) {
        /* subnormal range: quantum 2^-24; r == 1024 becomes the smallest normal */
        double r = rint(ldexp(a, 24)); /* exact scaling, then ties-to-even */
        return (uint16_t)(sign | (uint16_t)r);
    }
    double r = rint(ldexp(a, 10 - unbiased)); /* in [1024, 2048] */
    uint32_t bits = ((uint32_t)(unbiased + 15) << 10) + (uint32_t)(r - 1024.0);
    return (uint16_t)(sign | bits);            /* r == 2048 carries into the exponent */
}

void oracle_f16_to_f32_array(const uint16_t* in, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f32(in[i]);
}

void oracle_f32_to_f16_array(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Model-state memory per device.                                            */
/* ------------------------------------------------------------------------ */

/* Bytes of model state each device holds for Psi parameters, N_d ranks and an
 * optimizer-state multiplier K (12 for mixed-precision Adam):
 *   stage 0 (plain DP)            (4 + K) Psi
 *   stage 1 (optimizer states)    4 Psi + K Psi / N_d
 *   stage 2 (+ gradients)         2 Psi + (2 + K) Psi / N_d
 *   stage 3 (+ parameters)        (4 + K) Psi / N_d
 * ("DeepSpeed ZeRO Stages" sec. 1.2 and 3.1-3.3).  A stage outside 0..3 or
 * N_d < 1 gives NaN, standing in for the error the pages' Python raises. */
double oracle_state_bytes(double psi, int32_t n_d, int32_t stage, double k)
{
    if (n_d < 1) return NAN;
    double n = (double)n_d;
    switch (stage) {
    case 0: return (4.0 + k) * psi;
    case 1: return 4.0 * psi + k * psi / n;
    case 2: return 2.0 * psi + (2.0 + k) * psi / n;
    case 3: return (4.0 + k) * psi / n;
    default: return NAN;
    }
}

/* ------------------------------------------------------------------------ */
/* Partition of the flat parameter index set.                                */
/* ------------------------------------------------------------------------ */

typedef struct oracle_fragment {
    int32_t tensor;        /* tensor index in list order */
    int32_t shard;         /* owning rank */
    int64_t tensor_offset; /* first element of the fragment inside the tensor */
    int64_t shard_offset;  /* first element of the fragment inside the shard */
    int64_t length;        /* elements */
} oracle_fragment;

/* The tensors are packed back to back, in list order, into one flat buffer of
 * Psi elements.  The index set is padded to Psi_pad, the least multiple of
 * N_d * align, and split into N_d equal contiguous shards of S = Psi_pad / N_d
 * elements: shard i owns [i S, (i+1) S).  The shards are disjoint, their union
 * covers [0, Psi) and each holds about Psi / N_d real elements ("DeepSpeed
 * ZeRO Stages" sec. 2).  A fragment is the overlap of one tensor with one
 * shard; they are listed shard by shard, tensors in list order within a shard.
 *
 * frags == NULL asks for the count only.  Returns ORACLE_ERR_ARG (with
 * *n_frags set to the count needed) when frag_cap is too small. */
int32_t oracle_layout(const int64_t* numels, int32_t n_tensors, int32_t n_d, int32_t align,
                      int64_t* psi_out, int64_t* psi_pad_out, int64_t* shard_numel_out,
                      int64_t* tensor_offsets, int64_t* shard_offsets,
                      oracle_fragment* frags, int64_t frag_cap, int64_t* n_frags_out)
{
    if (n_tensors < 0 || n_d < 1 || align < 1 || (align & (align - 1)) != 0) return ORACLE_ERR_ARG;
    if (n_tensors > 0 && numels == NULL) return ORACLE_ERR_ARG;
    for (int32_t t = 0; t < n_tensors; ++t)
        if (numels[t] < 0) return ORACLE_ERR_ARG;

    /* exclusive prefix sum: where each tensor starts in the flat buffer */
    int64_t psi = 0;
    for (int32_t t = 0; t < n_tensors; ++t) {
        if (tensor_offsets) tensor_offsets[t] = psi;
        psi += numels[t];
    }
    int64_t unit = (int64_t)n_d * (int64_t)align;
    int64_t psi_pad = ((psi + unit - 1) / unit) * unit;
    int64_t s = psi_pad / n_d;
    if (psi_out) *psi_out = psi;
    if (psi_pad_out) *psi_pad_out = psi_pad;
    if (shard_numel_out) *shard_numel_out = s;
    if (shard_offsets)
        for (int32_t i = 0; i <= n_d; ++i) shard_offsets[i] = (int64_t)i * s;

    /* fragments: intersect every shard with every tensor */
    int64_t count = 0;
    for (int32_t i = 0; i < n_d; ++i) {
        int64_t shard_lo = (int64_t)i * s, shard_hi = shard_lo + s;
        int64_t start = 0;
        for (int32_t t = 0; t < n_tensors; ++t) {
            int64_t t_lo = start, t_hi = start + numels[t];
            start = t_hi;
            int64_t lo = t_lo > shard_lo ? t_lo : shard_lo;
            int64_t hi = t_hi < shard_hi ? t_hi : shard_hi;
            if (hi <= lo) continue;
            if (frags && count < frag_cap) {
                frags[count].tensor = t;
                frags[count].shard = i;
                frags[count].tensor_offset = lo - t_lo;
                frags[count].shard_offset = lo - shard_lo;
                frags[count].length = hi - lo;
            }
            ++count;
        }
    }
    if (n_frags_out) *n_frags_out = count;
    if (frags && count > frag_cap) return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Simulated reduce-scatter of the fp16 gradient contributions.              */
/* ------------------------------------------------------------------------ */

/* Rank i receives the gradient of its own shard "averaged" over the N_d ranks
 * ("ZeRO Stage 1 Math", "The per-step mechanics", beat 2).  contrib[k] points
 * at rank k's fp16 gradient for this shard (scaled by the loss scale L).
 *   gs_j = sum over k = 0..N_d-1, in that order, of fp32(h_k[j])
 *   g_j  = gs_j * (float)(1 / (N_d * L))
 * *nonfinite is set to 1 when some gs_j with j < n is not finite, else 0.
 * g may be NULL when only the overflow test is wanted. */
int32_t oracle_grad_reduce(const uint16_t* const* contrib, int32_t n_d, int64_t n,
                           double loss_scale, float* g, int32_t* nonfinite)
{
    if (n_d < 1 || n < 0 || !(loss_scale > 0.0) || contrib == NULL || nonfinite == NULL)
        return ORACLE_ERR_ARG;
    float inv = (float)(1.0 / ((double)n_d * loss_scale));
    int32_t bad = 0;
    for (int64_t j = 0; j < n; ++j) {
        float gs = 0.0f;
        for (int32_t k = 0; k < n_d; ++k) gs = gs + oracle_f16_to_f32(contrib[k][j]);
        if (!isfinite(gs)) bad = 1;
        if (g) g[j] = gs * inv;
    }
    *nonfinite = bad;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Adam / AdamW on the shard, then the fp16 cast.                            */
/* ------------------------------------------------------------------------ */

/* One update at Adam time t = step (>= 1) for n coordinates, in place on the
 * fp32 master theta, m and v, writing fp16(theta') into params:
 *   m'  = b1 m + (1 - b1) g
 *   v'  = b2 v + (1 - b2) g^2
 *   mh  = m' / (1 - beta1^t),  vh = v' / (1 - beta2^t)
 *   u   = mh / (sqrt(vh) + eps)
 *   th' = th - lr (u + wd th)           (wd = 0: plain Adam)
 *   p   = fp16(th')
 * ("DeepSpeed ZeRO Stages" sec. 2.1 Fact 1; "ZeRO Stage 1 Math", "Where the
 * 12 bytes come from"; decoupled decay for the AdamW optimizer type named in
 * "DeepSpeed ZeRO: Extreme Memory Efficiency", configuration example.) */
int32_t oracle_adam_apply(const float* g, int64_t n, float* master, float* m, float* v,
                          uint16_t* params, double lr, double beta1, double beta2,
                          double eps, double weight_decay, int64_t step)
{
    if (n < 0 || step < 1) return ORACLE_ERR_ARG;
    if (n > 0 && (g == NULL || master == NULL || m == NULL || v == NULL)) return ORACLE_ERR_ARG;

    double p1 = 1.0, p2 = 1.0;
    for (int64_t i = 0; i < step; ++i) {
        p1 = p1 * beta1;
        p2 = p2 * beta2;
    }
    float b1 = (float)beta1, c1 = (float)(1.0 - beta1);
    float b2 = (float)beta2, c2 = (float)(1.0 - beta2);
    float bc1 = (float)(1.0 - p1), bc2 = (float)(1.0 - p2);
    float lr_f = (float)lr, eps_f = (float)eps, wd_f = (float)weight_decay;

    for (int64_t j = 0; j < n; ++j) {
        float gj = g[j];
        float mj = b1 * m[j] + c1 * gj;
        float vj = b2 * v[j] + c2 * (gj * gj);
        float mh = mj / bc1;
        float vh = vj / bc2;
        float u = mh / (sqrtf(vh) + eps_f);
        float th = master[j];
        float th_new = th - lr_f * (u + wd_f * th);
        m[j] = mj;
        v[j] = vj;
        master[j] = th_new;
        if (params) params[j] = oracle_f32_to_f16(th_new);
    }
    return ORACLE_OK;
}

/* One whole shard step: reduce, test, and update only when every reduced
 * gradient is finite.  On overflow nothing is written and *overflow = 1.
 * scratch must hold n floats.  ("ZeRO Stage 1 Math", "The per-step
 * mechanics", beats 2-3; the skip is the dynamic loss-scale rule, which the
 * pages do not describe.) */
int32_t oracle_shard_step(const uint16_t* const* contrib, int32_t n_d, int64_t n,
                          float* master, float* m, float* v, uint16_t* params,
                          double lr, double beta1, double beta2, double eps,
                          double weight_decay, double loss_scale, int64_t step,
                          float* scratch, int32_t* overflow)
{
    if (overflow == NULL || (n > 0 && scratch == NULL)) return ORACLE_ERR_ARG;
    int32_t bad = 0;
    int32_t rc = oracle_grad_reduce(contrib, n_d, n, loss_scale, scratch, &bad);
    if (rc != ORACLE_OK) return rc;
    *overflow = bad;
    if (bad) return ORACLE_OK;
    return oracle_adam_apply(scratch, n, master, m, v, params, lr, beta1, beta2, eps,
                             weight_decay, step);
}

/* Bookkeeping after the overflow test of one step (over every shard stepped):
 * overflow -> the step is skipped, the loss scale halves (never below 1) and
 * the Adam time does not advance; otherwise the update is committed and the
 * count of applied updates grows by one.  (The usual dynamic loss-scale rule;
 * the pages do not describe loss scaling.  The Adam time t is the one of the
 * bias correction, "DeepSpeed ZeRO Stages", sec. 2.1, Fact 1.) */
void oracle_commit(int32_t overflow, double* loss_scale, int64_t* applied_steps)
{
    if (overflow) {
        double half = *loss_scale * 0.5;
        *loss_scale = half < 1.0 ? 1.0 : half;
    } else {
        *applied_steps += 1;
    }
}

/* ------------------------------------------------------------------------ */
/* Global gradient-norm clipping.                                            */
/* ------------------------------------------------------------------------ */

/* Adds sum_j g_j^2 over n reduced gradients to *sqnorm, in double, in index
 * order.  (A float squared is exact in double.)  Clipping couples every
 * coordinate through ||g||_2 over all of P ("DeepSpeed ZeRO Stages",
 * sec. 2.1, Fact 1), so each rank adds its shard and the ranks sum. */
void oracle_grad_sqnorm(const float* g, int64_t n, double* sqnorm)
{
    double acc = *sqnorm;
    for (int64_t j = 0; j < n; ++j) acc = acc + (double)g[j] * (double)g[j];
    *sqnorm = acc;
}

/* Clip factor for a global squared norm: min(1, max_norm / (||g|| + 1e-6)),
 * formed in double and rounded once to float.  max_norm <= 0 disables
 * clipping (factor 1).  ("DeepSpeed ZeRO Stages", sec. 2.1, Fact 1 names the
 * clipping; the formula is the common one, the pages give none.) */
float oracle_clip_factor(double sqnorm, double max_norm)
{
    if (!(max_norm > 0.0)) return 1.0f;
    double c = max_norm / (sqrt(sqnorm) + 1e-6);
    if (!(c < 1.0)) c = 1.0;
    return (float)c;
}

/* g_j <- g_j * c in fp32 (the clipped gradient; "DeepSpeed ZeRO Stages",
 * sec. 2.1, Fact 1). */
void oracle_scale(float* g, int64_t n, float c)
{
    for (int64_t j = 0; j < n; ++j) g[j] = g[j] * c;
}

/* ------------------------------------------------------------------------ */
/* Quantized parameter all-gather (ZeRO++ qwZ).                              */
/* ------------------------------------------------------------------------ */

#define ORACLE_QWZ_BLOCK 256

/* Block-wise symmetric int8 quantization of n fp16 parameters: for each block
 * of 256 consecutive values (the last one may be shorter) scale = max|x| / 127
 * and q = rint(x / scale), both in fp32 ("ZeRO Optimization: Stages 1, 2, and
 * 3 Explained", ZeRO++: 16-bit parameters sent as 8-bit with a scale per
 * small block).  codes[n], scales[ceil(n / 256)]. */
void oracle_qwz_quantize(const uint16_t* params, int64_t n, int8_t* codes, float* scales)
{
    for (int64_t b = 0; b * ORACLE_QWZ_BLOCK < n; ++b) {
        int64_t lo = b * ORACLE_QWZ_BLOCK;
        int64_t hi = lo + ORACLE_QWZ_BLOCK < n ? lo + ORACLE_QWZ_BLOCK : n;
        float amax = 0.0f;
        for (int64_t j = lo; j < hi; ++j) {
            float a = fabsf(oracle_f16_to_f32(params[j]));
            if (a > amax) amax = a;
        }
        float scale = amax / 127.0f;
        scales[b] = scale;
        for (int64_t j = lo; j < hi; ++j) {
            float q = 0.0f;
            if (scale > 0.0f) q = rintf(oracle_f16_to_f32(params[j]) / scale);
            if (q > 127.0f) q = 127.0f;
            if (q < -127.0f) q = -127.0f;
            codes[j] = (int8_t)q;
        }
    }
}

/* The receiver's side of the quantized all-gather: params[j] =
 * fp16(q_j * scale_of_its_block) ("ZeRO Optimization: Stages 1, 2, and 3
 * Explained", ZeRO++ quantized weights). */
void oracle_qwz_dequantize(const int8_t* codes, const float* scales, int64_t n, uint16_t* params)
{
    for (int64_t j = 0; j < n; ++j)
        params[j] = oracle_f32_to_f16((float)codes[j] * scales[j / ORACLE_QWZ_BLOCK]);
}

/* ------------------------------------------------------------------------ */
/* SGD with momentum.                                                        */
/* ------------------------------------------------------------------------ */

/* Mixed-precision SGD with momentum on n coordinates, in place on the fp32
 * master theta and momentum b, writing fp16(theta') into params:
 *   d  = g + wd theta          (L2 weight decay folded into the gradient)
 *   b' = mu b + d              (b starts at 0)
 *   th'= theta - lr b'
 * The pages name this optimizer through its state multiplier K ("DeepSpeed
 * ZeRO Stages" sec. 1.2) and give no formula; this is the textbook rule. */
int32_t oracle_sgd_apply(const float* g, int64_t n, float* master, float* mom, uint16_t* params,
                         double lr, double momentum, double weight_decay)
{
    if (n < 0 || (n > 0 && (g == NULL || master == NULL || mom == NULL))) return ORACLE_ERR_ARG;
    float lr_f = (float)lr, mu = (float)momentum, wd_f = (float)weight_decay;
    for (int64_t j = 0; j < n; ++j) {
        float th = master[j];
        float d = g[j] + wd_f * th;
        float b = mu * mom[j] + d;
        float th_new = th - lr_f * b;
        mom[j] = b;
        master[j] = th_new;
        if (params) params[j] = oracle_f32_to_f16(th_new);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* 8-bit Adam: m and v stored as 8-bit codes with a scale per block.         */
/* ------------------------------------------------------------------------ */

/* The pages name "8-bit Adam" only through its state multiplier K = 6
 * ("DeepSpeed ZeRO Stages" sec. 1.2): an fp32 master (4 bytes) and one byte
 * each for m and v.  The method followed is the block-wise 8-bit Adam of
 * Dettmers, Lewis, Shleifer and Zettlemoyer, "8-bit Optimizers via Block-wise
 * Quantization" (ICLR 2022): the states are cut into blocks of 2048
 * consecutive elements, each block keeps its largest magnitude as its scale,
 * and every element keeps the code of the table value nearest to
 * state / scale, the table being their dynamic (decimal-exponent) map.  Each
 * step dequantizes, runs the fp32 Adam update and quantizes the new states
 * again. */

#define ORACLE_ADAM8_BLOCK 2048

/* Value of code k (0 <= k < 2^bits) of the dynamic map over [0, 1]: code 0
 * is 0; otherwise the run of leading zero bits of k in a field of `bits` bits
 * is the decimal exponent E, the first set bit is the indicator, and the
 * f bits below it (f = bits - E - 1) pick one of F = 2^f equal steps of the
 * fraction range [0.1, 1]; the value is 10^-E * (0.1 + 0.9 (j + 1) / F) for
 * those bits j, formed in double in that order and rounded once to float.
 * (Reading: the fraction values are the upper ends of the F steps, so the
 * block's largest magnitude, x = 1, is exact.) */
static float oracle_dyn_value(int k, int bits)
{
    if (k == 0) return 0.0f;
    int len = 0;
    while ((k >> len) != 0) ++len;       /* bit length of k */
    int e = bits - len;                  /* leading zeros: the decimal exponent */
    int f = len - 1;                     /* fraction bits below the indicator */
    int j = k - (1 << f);
    double p10 = 1.0;
    for (int i = 0; i < e; ++i) p10 = p10 * 10.0;
    double frac = 0.1 + 0.9 * ((double)(j + 1) / (double)(1 << f));
    return (float)(frac / p10);
}

/* The two code tables: mag7[128], the magnitudes of the signed map (a sign
 * bit and 7 magnitude bits, for m), and mag8[256], the unsigned map (8 bits,
 * for v >= 0). */
void oracle_adam8_maps(float* mag7, float* mag8)
{
    for (int k = 0; k < 128; ++k) mag7[k] = oracle_dyn_value(k, 7);
    for (int k = 0; k < 256; ++k) mag8[k] = oracle_dyn_value(k, 8);
}

/* Index of the table entry nearest to a (distances in double); of two
 * equally near entries the smaller one.  A NaN a gives 0. */
static int oracle_nearest(float a, const float* table, int count)
{
    int best = 0;
    double best_d = fabs((double)a - (double)table[0]);
    for (int k = 1; k < count; ++k) {
        double d = fabs((double)a - (double)table[k]);
        if (d < best_d) {
            best = k;
            best_d = d;
        }
    }
    return best;
}

/* Code of x in [-1, 1] under the signed map: bit 7 set for x < 0 (unless the
 * magnitude code is 0), bits 0-6 the code of |x| in mag7. */
uint8_t oracle_adam8_code_signed(float x, const float* mag7)
{
    int k = oracle_nearest(fabsf(x), mag7, 128);
    return (uint8_t)((x < 0.0f && k > 0) ? (0x80 | k) : k);
}

/* Code of x in [0, 1] under the unsigned map. */
uint8_t oracle_adam8_code_unsigned(float x, const float* mag8)
{
    return (uint8_t)oracle_nearest(x, mag8, 256);
}

/* One 8-bit Adam update at Adam time t = step (>= 1) for n coordinates, in
 * place on master, the codes and the per-block scales, writing fp16(theta')
 * into params.  For every block of 2048 consecutive elements (the last one may
 * be shorter), with scales sm, sv of the block:
 *   m   = (+-mag7[code & 127]) * sm      v = mag8[code] * sv
 *   m', v', theta' and the fp16 cast as in oracle_adam_apply
 *   sm' = max |m'| over the block        sv' = max v' over the block
 *   codes of x = m' / sm' and v' / sv', each one IEEE fp32 division (x = 0
 *   when the scale is 0); the division is monotone and sm' / sm' = 1, so x
 *   never leaves [-1, 1] and needs no clamp
 * Codes 0 with scale 0 stand for m = v = 0 before the first step. */
int32_t oracle_adam8_apply(const float* g, int64_t n, float* master, uint8_t* m_codes, uint8_t* v_codes,
                           float* m_scale, float* v_scale, uint16_t* params, double lr, double beta1,
                           double beta2, double eps, double weight_decay, int64_t step)
{
    if (n < 0 || step < 1) return ORACLE_ERR_ARG;
    if (n > 0 && (g == NULL || master == NULL || m_codes == NULL || v_codes == NULL || m_scale == NULL ||
                  v_scale == NULL))
        return ORACLE_ERR_ARG;
    float mag7[128], mag8[256];
    oracle_adam8_maps(mag7, mag8);

    double p1 = 1.0, p2 = 1.0;
    for (int64_t i = 0; i < step; ++i) {
        p1 = p1 * beta1;
        p2 = p2 * beta2;
    }
    float b1 = (float)beta1, c1 = (float)(1.0 - beta1);
    float b2 = (float)beta2, c2 = (float)(1.0 - beta2);
    float bc1 = (float)(1.0 - p1), bc2 = (float)(1.0 - p2);
    float lr_f = (float)lr, eps_f = (float)eps, wd_f = (float)weight_decay;

    float m_new[ORACLE_ADAM8_BLOCK], v_new[ORACLE_ADAM8_BLOCK];
    for (int64_t b = 0; b * ORACLE_ADAM8_BLOCK < n; ++b) {
        int64_t lo = b * ORACLE_ADAM8_BLOCK;
        int64_t hi = lo + ORACLE_ADAM8_BLOCK < n ? lo + ORACLE_ADAM8_BLOCK : n;
        float sm = m_scale[b], sv = v_scale[b];
        float amax_m = 0.0f, amax_v = 0.0f;
        for (int64_t j = lo; j < hi; ++j) {
            int cm = m_codes[j];
            float mag = mag7[cm & 0x7f];
            float m_old = ((cm & 0x80) ? -mag : mag) * sm;
            float v_old = mag8[v_codes[j]] * sv;
            float gj = g[j];
            float mj = b1 * m_old + c1 * gj;
            float vj = b2 * v_old + c2 * (gj * gj);
            float mh = mj / bc1;
            float vh = vj / bc2;
            float u = mh / (sqrtf(vh) + eps_f);
            float th = master[j];
            float th_new = th - lr_f * (u + wd_f * th);
            master[j] = th_new;
            if (params) params[j] = oracle_f32_to_f16(th_new);
            m_new[j - lo] = mj;
            v_new[j - lo] = vj;
            if (fabsf(mj) > amax_m) amax_m = fabsf(mj);
            if (vj > amax_v) amax_v = vj;
        }
        for (int64_t j = lo; j < hi; ++j) {
            float xm = amax_m > 0.0f ? m_new[j - lo] / amax_m : 0.0f;
            float xv = amax_v > 0.0f ? v_new[j - lo] / amax_v : 0.0f;
            m_codes[j] = oracle_adam8_code_signed(xm, mag7);
            v_codes[j] = oracle_adam8_code_unsigned(xv, mag8);
        }
        m_scale[b] = amax_m;
        v_scale[b] = amax_v;
    }
    return ORACLE_OK;
}
