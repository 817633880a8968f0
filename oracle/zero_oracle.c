/*
 * zero_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * A plain, slow, scalar CPU statement of what one ZeRO data-parallel rank
 * computes in its mixed-precision optimizer step.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or constant with the CUDA library; the two meet only
 * through the seeded synthetic inputs.
 *
 * Sources (web pages on ZeRO / DeepSpeed):
 *   [ZeRO card]  "ZeRO: Memory Optimizations Toward Training Trillion
 *                Parameter Models - 中文验证版" (ai-papers.xuzou.cn/zh/papers/zero_2019/)
 *                sections 瓶颈 (bottleneck), 方法适配 (method), 证据 (evidence).
 *   [DS news]    DeepSpeed release news (lxsoso.com/blog/19320.html): the engine
 *                manages mixed precision and gradient accumulation.
 *   [ZeRO-2]     "探秘微软大规模人工智能的新框架 ZeRO-2" (infoq.cn), section
 *                "Zero-2和DeepSpeed".
 *
 * What the pages fix: the model state of mixed-precision Adam is an fp16
 * parameter and gradient plus an fp32 copy of the parameter, the momentum and
 * the variance ([ZeRO card §瓶颈]); ZeRO splits these states over the Nd
 * data-parallel ranks instead of replicating them ([ZeRO card §方法适配]).
 * The arithmetic therefore runs in the precision of the fp32 state: every
 * per-element operation below is one IEEE binary32 operation, round to
 * nearest even, evaluated in source order with no contraction into FMA
 * (build with -ffp-contract=off, no fast-math).
 *
 * What the pages leave open, and the reading taken here:
 *   - the update is Adam (Kingma & Ba 2015, Algorithm 1) with decoupled
 *     weight decay (Loshchilov & Hutter 2019): with g the unscaled, clipped
 *     gradient and t the number of applied steps,
 *         m <- b1 m + (1-b1) g,   v <- b2 v + (1-b2) g^2,
 *         p <- p - lr ( m_hat / (sqrt(v_hat) + eps) + wd p ),
 *         m_hat = m / (1-b1^t),   v_hat = v / (1-b2^t);
 *     the two bias corrections are carried as per-step scalars
 *     lr/(1-b1^t) and 1/sqrt(1-b2^t) (the same quantity, regrouped);
 *   - dynamic loss scaling (Micikevicius et al. 2018, section 3.2): an
 *     inf/NaN anywhere in the gradient skips the step (no state changes, t
 *     unchanged) and halves the scale down to a floor; a run of
 *     `scale_window` clean steps doubles it;
 *   - the global gradient norm is the L2 norm of the unscaled, unclipped
 *     gradient over every shard; clipping multiplies g by
 *     max_norm / (norm + 1e-6) when that is below 1 and max_norm > 0;
 *   - every step scalar is computed in binary64 from binary64
 *     hyper-parameters and rounded once to binary32.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* Element encodings of a gradient or low-precision parameter array. */
enum { ZO_F16 = 0, ZO_BF16 = 1, ZO_F32 = 2 };

/* ---- scalar conversions ------------------------------------------------ */

static float f16_bits_to_f32(uint16_t bits)
{
    _Float16 h;
    memcpy(&h, &bits, sizeof h);
    return (float)h; /* exact: every binary16 value is a binary32 value */
}

static uint16_t f32_to_f16_bits(float x)
{
    _Float16 h = (_Float16)x; /* IEEE conversion, round to nearest even */
    uint16_t bits;
    memcpy(&bits, &h, sizeof bits);
    return bits;
}

static float bf16_bits_to_f32(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16; /* bfloat16 is the top half of binary32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even.  Adding
 * 0x7FFF + (bit 16) to the binary32 pattern carries into bit 16 exactly when
 * the dropped low half is above one half ulp, or equal to it with an odd
 * kept part; a carry out of the mantissa bumps the exponent, which is the
 * correct rounding (up to infinity for values past the largest bfloat16).
 * NaN keeps its sign and gets the quiet bit. */
static uint16_t f32_to_bf16_bits(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if (isnan(x))
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float load_elem(const void *buf, int dtype, int64_t i)
{
    switch (dtype) {
    case ZO_F16: return f16_bits_to_f32(((const uint16_t *)buf)[i]);
    case ZO_BF16: return bf16_bits_to_f32(((const uint16_t *)buf)[i]);
    default: return ((const float *)buf)[i];
    }
}

static void store_lp(void *buf, int dtype, int64_t i, float x)
{
    if (dtype == ZO_F16)
        ((uint16_t *)buf)[i] = f32_to_f16_bits(x);
    else
        ((uint16_t *)buf)[i] = f32_to_bf16_bits(x);
}

/* Exposed for the conversion pins (numpy's binary16 and torch's bfloat16
 * casts are the library special cases they are checked against). */
void zo_f32_to_lp(const float *x, void *out, int dtype, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        store_lp(out, dtype, i, x[i]);
}

void zo_lp_to_f32(const void *in, int dtype, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = load_elem(in, dtype, i);
}

/* ---- gradient accumulation ------------------------------------------- */

/* [DS news] "gradient accumulation": the gradients of n_bufs micro-batches
 * are summed into one fp32 buffer.  Reading: the sum runs in micro-batch order
 * k = 0, 1, ..., one binary32 addition at a time; with `overwrite` the sum
 * starts from float(g_0), otherwise from the current contents of acc. */
void zo_accumulate(float *acc, const void *const *bufs, int32_t n_bufs, int dtype,
                   int64_t n, int32_t overwrite)
{
    for (int64_t i = 0; i < n; ++i) {
        float a;
        int32_t k = 0;
        if (overwrite) {
            a = load_elem(bufs[0], dtype, i);
            k = 1;
        } else {
            a = acc[i];
        }
        for (; k < n_bufs; ++k)
            a = a + load_elem(bufs[k], dtype, i);
        acc[i] = a;
    }
}

/* ---- ZeRO stage 2: the gradient reduction onto the owned shard ------ */

/* [ZeRO card §方法适配] stage 2 partitions the gradients: each rank keeps
 * only the reduced gradient of its own shard, which the data-parallel
 * reduce-scatter delivers.  The arithmetic of that reduction, on one rank:
 *     out[i] = round( (g_0[i] + g_1[i] + ... + g_{Nd-1}[i]) / Nd )
 * Reading: binary32 sum in rank order starting from float(g_0[i]), one
 * IEEE binary32 division by Nd (the data-parallel mean), rounded to nearest
 * even into the output type (binary32 output is stored as is). */
void zo_reduce_mean(const void *const *bufs, int32_t n_bufs, int dtype, int64_t n, void *out,
                    int out_dtype)
{
    const float count = (float)n_bufs;
    for (int64_t i = 0; i < n; ++i) {
        float a = load_elem(bufs[0], dtype, i);
        for (int32_t k = 1; k < n_bufs; ++k)
            a = a + load_elem(bufs[k], dtype, i);
        const float mean = a / count;
        if (out_dtype == ZO_F32)
            ((float *)out)[i] = mean;
        else
            store_lp(out, out_dtype, i, mean);
    }
}

/* ---- pass 1: unscale, overflow, squared norm ------------------------- */

/* Adds sum_i g_i^2 into *sumsq, g_i = float(g_lp_i) * inv_scale (a binary32
 * product; exact for a power-of-two scale), squared and summed in binary64
 * in index order.  Sets *found_inf to 1 if any g_i is +-inf or NaN.  Called
 * once per array, in order, it folds several shards into one global sum. */
void zo_norm_overflow(const void *g, int dtype, int64_t n, float inv_scale,
                      double *sumsq, int32_t *found_inf)
{
    double s = *sumsq;
    int32_t bad = *found_inf;
    for (int64_t i = 0; i < n; ++i) {
        float gi = load_elem(g, dtype, i) * inv_scale;
        if (!isfinite(gi))
            bad = 1;
        s += (double)gi * (double)gi;
    }
    *sumsq = s;
    *found_inf = bad;
}

/* ---- the step decision and its scalars ------------------------------- */

typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    double max_norm;      /* <= 0: no clipping */
    double min_scale;     /* floor of the loss scale */
    int64_t scale_window; /* clean steps in a row before the scale doubles */
} zo_hparams;

typedef struct {
    double loss_scale;  /* S: gradients arrive multiplied by S */
    int64_t step;       /* t: steps applied so far */
    int64_t good_steps; /* clean steps since the scale last changed */
} zo_scaler;

typedef struct {
    float inv_scale, clip;
    float beta1, one_minus_beta1, beta2, one_minus_beta2, eps;
    float step_size;    /* lr / (1 - beta1^t) */
    float inv_sqrt_bc2; /* 1 / sqrt(1 - beta2^t) */
    float lr_wd;        /* lr * weight_decay */
    int32_t skip;
    double norm;
} zo_step;

/* Takes the global (sumsq, found_inf) of this step, decides skip or apply,
 * advances the loss scaler and fills the per-step scalars.  The scale used
 * to unscale this step's gradients is the one in force before the update. */
void zo_decide(const zo_hparams *hp, zo_scaler *sc, double sumsq, int32_t found_inf,
               zo_step *out)
{
    memset(out, 0, sizeof *out);
    out->inv_scale = (float)(1.0 / sc->loss_scale);
    out->norm = sqrt(sumsq);

    if (found_inf) {
        out->skip = 1;
        double s = sc->loss_scale / 2.0;
        sc->loss_scale = s < hp->min_scale ? hp->min_scale : s;
        sc->good_steps = 0;
        out->clip = 1.0f;
        return;
    }

    sc->step += 1;
    sc->good_steps += 1;
    if (sc->good_steps >= hp->scale_window) {
        sc->loss_scale *= 2.0;
        sc->good_steps = 0;
    }

    double clip = 1.0;
    if (hp->max_norm > 0.0) {
        double c = hp->max_norm / (out->norm + 1e-6);
        if (c < 1.0)
            clip = c;
    }
    const double t = (double)sc->step;
    const double bc1 = 1.0 - pow(hp->beta1, t);
    const double bc2 = 1.0 - pow(hp->beta2, t);

    out->clip = (float)clip;
    out->beta1 = (float)hp->beta1;
    out->one_minus_beta1 = (float)(1.0 - hp->beta1);
    out->beta2 = (float)hp->beta2;
    out->one_minus_beta2 = (float)(1.0 - hp->beta2);
    out->eps = (float)hp->eps;
    out->step_size = (float)(hp->lr / bc1);
    out->inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));
    out->lr_wd = (float)(hp->lr * hp->weight_decay);
    out->skip = 0;
}

/* ---- pass 2: clip, AdamW, cast --------------------------------------- */

/* One element, in binary32:
 *     g  = float(g_lp) * inv_scale;  g = g * clip   (clip below 1 only)
 *     m' = b1*m + (1-b1)*g
 *     v' = b2*v + (1-b2)*(g*g)
 *     u  = m' / (sqrt(v') * inv_sqrt_bc2 + eps)
 *     p' = p - (step_size*u + lr_wd*p)      decoupled decay on the old p
 * The caller rounds p' to nearest even in the low-precision type. */
static void adam_element(float g_lp, float *p, float *m, float *v, const zo_step *s)
{
    float g = g_lp * s->inv_scale;
    if (s->clip != 1.0f)
        g = g * s->clip;
    float m1 = s->beta1 * *m + s->one_minus_beta1 * g;
    float v1 = s->beta2 * *v + s->one_minus_beta2 * (g * g);
    float denom = sqrtf(v1) * s->inv_sqrt_bc2 + s->eps;
    float u = m1 / denom;
    float p1 = *p - (s->step_size * u + s->lr_wd * *p);
    *m = m1;
    *v = v1;
    *p = p1;
}

/* The update over whole arrays.  A skipped step touches nothing. */
void zo_adam_apply(const void *g, int gdtype, float *p, float *m, float *v, void *p_lp,
                   int pdtype, int64_t n, const zo_step *s)
{
    if (s->skip)
        return;
    for (int64_t i = 0; i < n; ++i) {
        adam_element(load_elem(g, gdtype, i), &p[i], &m[i], &v[i], s);
        if (p_lp)
            store_lp(p_lp, pdtype, i, p[i]);
    }
}

/* The same update on gathered elements: idx[j] names an element of the full
 * gradient array, the state arrays hold only the gathered elements.  Lets a
 * test follow a sample of a shard too large to update whole on the host. */
void zo_adam_apply_sampled(const void *g, int gdtype, const int64_t *idx, float *p, float *m,
                           float *v, void *p_lp, int pdtype, int64_t n_samples, const zo_step *s)
{
    if (s->skip)
        return;
    for (int64_t j = 0; j < n_samples; ++j) {
        adam_element(load_elem(g, gdtype, idx[j]), &p[j], &m[j], &v[j], s);
        if (p_lp)
            store_lp(p_lp, pdtype, j, p[j]);
    }
}

/* ---- 1-bit Adam: the compression stage ------------------------------- */

/* [DS news] names 1-bit Adam: Adam with up to 5x less communication and
 * Adam's convergence, 3.5x faster where communication is the bottleneck.
 * The pages give no algorithm.  The reading follows the outline of the
 * published method (Tang et al. 2021, "1-bit Adam: Communication Efficient
 * Large-Scale Training with Adam's Convergence Speed"):
 *   - a warm-up of T_w steps of plain Adam (zo_adam_apply above);
 *   - then the variance is frozen at its value after step T_w, and with it
 *     its bias correction 1/sqrt(1 - b2^T_w); each worker i updates its
 *     momentum locally from the last synchronised momentum m,
 *         m_i = b1*m + (1-b1)*g_i        (g_i unscaled and clipped as above),
 *     and the workers average their momenta through a compressed all-reduce
 *     with error feedback at both ends:
 *       worker i:  x = m_i + e_i;  c_i = C(x);  e_i <- x - c_i
 *                  (chunk j of c_i's signs and its scale go to rank j);
 *       rank j:    y = (sum over i of c_i on chunk j) / Nd + f_j;
 *                  s_j = C(y);  f_j <- y - s_j  (s_j goes to every worker);
 *       worker:    m = the concatenation of the s_j, the new synchronised
 *                  momentum, and
 *                  p <- p - (lr/(1-b1^t) * m / (sqrt(v) * isb2(T_w) + eps) + lr*wd*p).
 * Choices the outline leaves open, made here: the 1-bit compressor is
 * C(x) = scale * sign(x) with scale = ||x||_2 / sqrt(n) (the compressed
 * vector keeps x's L2 norm) and sign(0) = sign(-0) = +1; the squared norm is
 * summed in binary64 in index order and scale = sqrt(sum / n) is rounded
 * once to binary32; the server's average is the binary32 sum of the Nd
 * worker values in rank order followed by one division by Nd; the signs
 * travel as bits, bit k of 32-bit word w holding element 32w + k, 1 for +.
 * Binary32 with one rounding per operation, as everywhere in this file. */

/* C applied in place: buf holds x on entry and the new error x - C(x) on
 * return; the signs go to bits and the scale to *scale.  A scale_in >= 0
 * replaces the computed scale (a test then follows another implementation's
 * rounding of the norm).  x_out, if not NULL, receives x itself (for
 * implementations that keep x and its scale and form the error x - C(x)
 * when they next read it). */
static void onebit_compress(float *buf, int64_t n, uint32_t *bits, float *scale, float scale_in, float *x_out)
{
    if (x_out)
        for (int64_t i = 0; i < n; ++i)
            x_out[i] = buf[i];
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i)
        s += (double)buf[i] * (double)buf[i];
    const float sc = scale_in >= 0.0f ? scale_in : (float)sqrt(s / (double)n);
    for (int64_t w = 0; w < (n + 31) / 32; ++w)
        bits[w] = 0u;
    for (int64_t i = 0; i < n; ++i) {
        const int plus = !(buf[i] < 0.0f);
        if (plus)
            bits[i / 32] |= 1u << (i % 32);
        buf[i] = buf[i] - (plus ? sc : -sc);
    }
    *scale = sc;
}

/* Worker i: local momentum from the synchronised m, error feedback and
 * compression.  e (the worker's error, n elements) is updated; m is read
 * only.  A skipped step touches nothing. */
void zo_onebit_worker(const void *g, int gdtype, int64_t n, const zo_step *s, const float *m,
                      float *e, uint32_t *bits, float *scale, float scale_in, float *x_out)
{
    if (s->skip)
        return;
    for (int64_t i = 0; i < n; ++i) {
        float gi = load_elem(g, gdtype, i) * s->inv_scale;
        if (s->clip != 1.0f)
            gi = gi * s->clip;
        const float mi = s->beta1 * m[i] + s->one_minus_beta1 * gi;
        e[i] = mi + e[i];
    }
    onebit_compress(e, n, bits, scale, scale_in, x_out);
}

/* Rank j as the server of its chunk of S elements: the Nd workers' signs
 * on that chunk (bits[i]: S/32 words) with their scales, averaged, plus the
 * server error f (S elements, updated), compressed again. */
void zo_onebit_server(const uint32_t *const *bits, const float *scales, int32_t nd, int64_t S,
                      float *f, uint32_t *out_bits, float *out_scale, float scale_in, int32_t skip,
                      float *x_out)
{
    if (skip)
        return;
    const float count = (float)nd;
    for (int64_t i = 0; i < S; ++i) {
        float a = 0.0f;
        for (int32_t k = 0; k < nd; ++k) {
            const float c = ((bits[k][i / 32] >> (i % 32)) & 1u) ? scales[k] : -scales[k];
            a = k == 0 ? c : a + c;
        }
        f[i] = a / count + f[i];
    }
    onebit_compress(f, S, out_bits, out_scale, scale_in, x_out);
}

/* Every worker: the synchronised momentum from the servers' signs (bits:
 * n/32 words, n = Nd*S, chunk j from rank j) and scales over the whole
 * padded buffer (the compressed all-reduce runs over all n elements), then
 * the parameter update with the frozen variance for the first `numel`
 * elements (the rest of the padded buffer is not parameters). */
void zo_onebit_update(const uint32_t *bits, const float *scales, int64_t S, int64_t n, int64_t numel,
                      float *p, float *m, const float *v, void *p_lp, int pdtype, const zo_step *s)
{
    if (s->skip)
        return;
    for (int64_t i = 0; i < n; ++i) {
        const float sc = scales[i / S];
        const float mi = ((bits[i / 32] >> (i % 32)) & 1u) ? sc : -sc;
        m[i] = mi;
        if (i >= numel)
            continue;
        const float denom = sqrtf(v[i]) * s->inv_sqrt_bc2 + s->eps;
        const float u = mi / denom;
        p[i] = p[i] - (s->step_size * u + s->lr_wd * p[i]);
        if (p_lp)
            store_lp(p_lp, pdtype, i, p[i]);
    }
}
