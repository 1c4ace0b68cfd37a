/*
 * oracle.c -- CPU definitions of the three fused memory-bound chains.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Plain loops in the order the
 * pages write the formulas; no blocking, no fusion, no reordering.  Build with
 * -O2 -ffp-contract=off and without -ffast-math, so each fp32 operation below
 * is rounded on its own exactly as an eager fp32 tensor op would round it.
 *
 * Precision readings (where the pages do not fix a step, the plainest reading
 * that the rest of the page supports):
 *   o1  The pages' chain runs on fp32 tensors, one rounded op at a time
 *       ([P1] §3.1 baseline: add, relu, mul, add), so the oracle is that fp32
 *       sequence.  The bf16 variant widens its inputs, runs the same fp32
 *       sequence and rounds the result once to bf16.
 *   o2  The [P4] example is fp32 ("x is f32[1024, 1024]"): every pointwise op
 *       is an fp32 op.  The row mean is a sum then a division by the row
 *       length ([P4] §6.4: the reduction is a 'sum', the /1024 happens in the
 *       consumer); the order of that sum is unspecified, so the oracle sums in
 *       double and rounds the mean once to fp32.
 *   o3  v = x + r is the fp32 add of the [P2] §2.3 kernel; the statistics,
 *       normalisation, affine step and GeLU are evaluated in double (the
 *       pages' rsqrtf / tanhf and one-pass E[v^2]-mean^2 are shortcuts of the
 *       fp32 sketch, not the definition), and the output is rounded once.
 *   o4  The LayerNorm family follows o3 with the residual optional, the
 *       residual sum optionally written out (rounded once to the I/O type) and
 *       the activation chosen (none, relu, gelu-tanh).
 *   o5  Row softmax in double, relative to the row maximum, rounded once.
 *   o6  Dropout ([P2] §2.1 LayerNorm -> ReLU -> Dropout): the pages fix no
 *       random number generator, so the decision of element i comes from the
 *       published Philox-4x32-10 counter-based generator at a counter fixed by
 *       (offset, i) and a key fixed by seed, one 16-bit uniform per element
 *       (eight per generator block); kept elements are scaled by 1 / (1 - p)
 *       in double, dropped ones are the product with 0.
 */
#include "oracle.h"

#include <math.h>
#include <string.h>

static const double ORACLE_PI = 3.14159265358979323846264338327950288;

/* ------------------------------------------------------------------------ */
/* scalar helpers                                                           */
/* ------------------------------------------------------------------------ */

float oracle_relu_f32(float v)
{
    /* [P1] §3.2 applies fmaxf(v, 0.0f).  v > 0 keeps v; every other value,
     * including -0 and NaN, becomes +0. */
    if (v > 0.0f)
        return v;
    return 0.0f;
}

double oracle_gelu_tanh(double z)
{
    /* [P2] §2.3: 0.5 * n * (1 + tanh(0.7978845608 * (n + 0.044715 * n^3)));
     * 0.7978845608 is sqrt(2/pi) to ten digits. */
    const double k = sqrt(2.0 / ORACLE_PI);
    double u = k * (z + 0.044715 * z * z * z);
    return 0.5 * z * (1.0 + tanh(u));
}

double oracle_bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

uint16_t oracle_bf16_from_double(double v)
{
    /* bf16: 1 sign bit, 8 exponent bits (bias 127), 7 stored fraction bits.
     * The value is rounded once, to the nearest multiple of the bf16 quantum
     * at its binade, ties to even (rint in the default rounding mode). */
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;

    int e;
    (void)frexp(a, &e);            /* a = f * 2^e, 0.5 <= f < 1           */
    int q = e - 8;                 /* 8 significant bits: quantum 2^(e-8) */
    if (q < -133)                  /* below 2^-126: fixed subnormal step   */
        q = -133;
    double k = rint(ldexp(a, -q)); /* exact scaling, one rounding          */
    double r = ldexp(k, q);
    if (r >= ldexp(1.0, 128))      /* rounded past the largest finite     */
        return (uint16_t)(sign | 0x7F80u);

    float rf = (float)r;           /* exact: r has <= 8 significant bits   */
    uint32_t bits;
    memcpy(&bits, &rf, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

static float widen_bf16(uint16_t h)
{
    return (float)oracle_bf16_to_double(h);
}

/* ------------------------------------------------------------------------ */
/* o1: y = relu(x + b1) * scale + b2                                        */
/* [P1] §1.1 (the four eager steps) and §3.1 (the baseline function)        */
/* ------------------------------------------------------------------------ */

static float o1_element(float x, float b1, float b2, float scale)
{
    float tmp = x + b1;             /* step 1: x + b1    -> tmp1 */
    tmp = oracle_relu_f32(tmp);     /* step 2: relu      -> tmp2 */
    tmp = tmp * scale;              /* step 3: * scale   -> tmp3 */
    tmp = tmp + b2;                 /* step 4: + b2      -> y    */
    return tmp;
}

void oracle_add_relu_scale_f32(const float *x, const float *b1, const float *b2,
                               float *y, int64_t n, float scale)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = o1_element(x[i], b1[i], b2[i], scale);
}

void oracle_add_relu_scale_bf16(const uint16_t *x, const uint16_t *b1,
                                const uint16_t *b2, uint16_t *y, int64_t n,
                                float scale)
{
    for (int64_t i = 0; i < n; ++i) {
        float r = o1_element(widen_bf16(x[i]), widen_bf16(b1[i]),
                             widen_bf16(b2[i]), scale);
        y[i] = oracle_bf16_from_double((double)r);
    }
}

/* o1 over rows x cols with b1 and/or b2 given per column (a length-cols
 * vector broadcast over the rows, as a bias is) */
static float o1_operand(const void *v, int bf16, int per_col, int64_t i, int64_t j,
                        int64_t cols)
{
    int64_t k = per_col ? j : i * cols + j;
    return bf16 ? widen_bf16(((const uint16_t *)v)[k]) : ((const float *)v)[k];
}

static void o1_bcast(const void *x, const void *b1, const void *b2, void *y, int bf16,
                     int64_t rows, int64_t cols, int b1_per_col, int b2_per_col, float scale)
{
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t j = 0; j < cols; ++j) {
            float xv = o1_operand(x, bf16, 0, i, j, cols);
            float r = o1_element(xv, o1_operand(b1, bf16, b1_per_col, i, j, cols),
                                 o1_operand(b2, bf16, b2_per_col, i, j, cols), scale);
            if (bf16)
                ((uint16_t *)y)[i * cols + j] = oracle_bf16_from_double((double)r);
            else
                ((float *)y)[i * cols + j] = r;
        }
    }
}

void oracle_add_relu_scale_bcast_f32(const float *x, const float *b1, const float *b2,
                                     float *y, int64_t rows, int64_t cols, int b1_per_col,
                                     int b2_per_col, float scale)
{
    o1_bcast(x, b1, b2, y, 0, rows, cols, b1_per_col, b2_per_col, scale);
}

void oracle_add_relu_scale_bcast_bf16(const uint16_t *x, const uint16_t *b1,
                                      const uint16_t *b2, uint16_t *y, int64_t rows,
                                      int64_t cols, int b1_per_col, int b2_per_col, float scale)
{
    o1_bcast(x, b1, b2, y, 1, rows, cols, b1_per_col, b2_per_col, scale);
}

/* ------------------------------------------------------------------------ */
/* o2: TorchInductor example chain, [P4] "model" and Figure 1               */
/* ------------------------------------------------------------------------ */

static float o2_s(float x, float bias, float x_scale, float branch_scale)
{
    float t = x * x_scale;          /* t = x * 1.1 + bias (broadcast bias) */
    t = t + bias;
    float a = oracle_relu_f32(t);   /* a = relu(t)                          */
    float p = a * a;                /* p = a * a                            */
    float q = a * branch_scale;     /* q = a * 0.1                          */
    float s = p + q;                /* s = p + q                            */
    return s;
}

void oracle_bias_relu_branch_mean_epilogue(const float *x, const float *bias,
                                           const float *gamma, const float *beta,
                                           float *y, int64_t rows, int64_t cols,
                                           float x_scale, float branch_scale,
                                           float *s_out, float *m_out)
{
    for (int64_t i = 0; i < rows; ++i) {
        const float *xr = x + i * cols;

        /* m = s.mean(dim=1, keepdim=True): row sum, then / cols */
        double sum = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            sum += (double)o2_s(xr[j], bias[j], x_scale, branch_scale);
        float m = (float)(sum / (double)cols);
        if (m_out)
            m_out[i] = m;

        /* y = (s - m) * gamma + beta */
        for (int64_t j = 0; j < cols; ++j) {
            float s = o2_s(xr[j], bias[j], x_scale, branch_scale);
            if (s_out)
                s_out[i * cols + j] = s;
            float d = s - m;
            d = d * gamma[j];
            y[i * cols + j] = d + beta[j];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* o3: residual + LayerNorm + affine + GeLU-tanh                            */
/* [P2] §2.2-2.3 (fused kernel: v = x + residual, mean, var, rsqrt(var+eps),*/
/* norm = (v-mean)*inv_std*weight + bias, GeLU) and [P3] §4.3 (two-pass     */
/* variance sum((x-mean)^2)/cols, rsqrt(var + eps), * gamma + beta)         */
/* ------------------------------------------------------------------------ */

typedef float (*o3_load_fn)(const void *p, int64_t i);

static float load_f32(const void *p, int64_t i) { return ((const float *)p)[i]; }
static float load_bf16(const void *p, int64_t i)
{
    return widen_bf16(((const uint16_t *)p)[i]);
}

static void o3_rows(const void *x, const void *r, const void *w, const void *b,
                    o3_load_fn load, void *out, int out_bf16, int64_t rows,
                    int64_t hidden, float eps, double *mean_out,
                    double *rstd_out, double *xhat_out)
{
    for (int64_t i = 0; i < rows; ++i) {
        int64_t base = i * hidden;

        /* mean = sum(v) / H, v = x + r in fp32 */
        double sum = 0.0;
        for (int64_t j = 0; j < hidden; ++j) {
            float v = load(x, base + j) + load(r, base + j);
            sum += (double)v;
        }
        double mean = sum / (double)hidden;

        /* var = sum((v - mean)^2) / H  (biased, two passes) */
        double sq = 0.0;
        for (int64_t j = 0; j < hidden; ++j) {
            float v = load(x, base + j) + load(r, base + j);
            double d = (double)v - mean;
            sq += d * d;
        }
        double var = sq / (double)hidden;
        double rstd = 1.0 / sqrt(var + (double)eps);
        if (mean_out)
            mean_out[i] = mean;
        if (rstd_out)
            rstd_out[i] = rstd;

        /* n = (v - mean) * rstd * w + b;  out = gelu_tanh(n) */
        for (int64_t j = 0; j < hidden; ++j) {
            float v = load(x, base + j) + load(r, base + j);
            double xhat = ((double)v - mean) * rstd;
            if (xhat_out)
                xhat_out[base + j] = xhat;
            double n = xhat * (double)load(w, j) + (double)load(b, j);
            double g = oracle_gelu_tanh(n);
            if (out_bf16)
                ((uint16_t *)out)[base + j] = oracle_bf16_from_double(g);
            else
                ((float *)out)[base + j] = (float)g;
        }
    }
}

void oracle_residual_layernorm_gelu_f32(const float *x, const float *r,
                                        const float *w, const float *b,
                                        float *out, int64_t rows, int64_t hidden,
                                        float eps, double *mean_out,
                                        double *rstd_out, double *xhat_out)
{
    o3_rows(x, r, w, b, load_f32, out, 0, rows, hidden, eps, mean_out,
            rstd_out, xhat_out);
}

void oracle_residual_layernorm_gelu_bf16(const uint16_t *x, const uint16_t *r,
                                         const uint16_t *w, const uint16_t *b,
                                         uint16_t *out, int64_t rows,
                                         int64_t hidden, float eps,
                                         double *mean_out, double *rstd_out,
                                         double *xhat_out)
{
    o3_rows(x, r, w, b, load_bf16, out, 1, rows, hidden, eps, mean_out,
            rstd_out, xhat_out);
}

/* ------------------------------------------------------------------------ */
/* o2 with bf16 I/O                                                         */
/* ------------------------------------------------------------------------ */

void oracle_bias_relu_branch_mean_epilogue_bf16(const uint16_t *x, const uint16_t *bias,
                                                const uint16_t *gamma, const uint16_t *beta,
                                                uint16_t *y, int64_t rows, int64_t cols,
                                                float x_scale, float branch_scale)
{
    for (int64_t i = 0; i < rows; ++i) {
        const uint16_t *xr = x + i * cols;
        double sum = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            sum += (double)o2_s(widen_bf16(xr[j]), widen_bf16(bias[j]), x_scale,
                                branch_scale);
        float m = (float)(sum / (double)cols);
        for (int64_t j = 0; j < cols; ++j) {
            float s = o2_s(widen_bf16(xr[j]), widen_bf16(bias[j]), x_scale, branch_scale);
            float d = s - m;
            d = d * widen_bf16(gamma[j]);
            float o = d + widen_bf16(beta[j]);
            y[i * cols + j] = oracle_bf16_from_double((double)o);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* o6: counter-based random numbers and the dropout decision                */
/* "Parallel random numbers: as easy as 1, 2, 3" (Salmon, Moraes, Dror and */
/* Shaw, SC'11), the Philox-4xW-10 generator: a counter of four W-bit words */
/* and a key of two; each of ten rounds multiplies counter words 0 and 2 by */
/* the round multipliers M0 and M1 (full 2W-bit products) and forms         */
/*   (hi(M1 c2) ^ c1 ^ k0,  lo(M1 c2),  hi(M0 c0) ^ c3 ^ k1,  lo(M0 c0)),     */
/* and before every round but the first the key words are bumped by the    */
/* Weyl constants W0, W1 (the leading W bits of the golden ratio's fraction */
/* and of sqrt(3) - 1).  The pages use dropout but fix no generator.        */
/* ------------------------------------------------------------------------ */

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += W0;
            k1 += W1;
        }
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += W0;
            k1 += W1;
        }
        unsigned __int128 p0 = (unsigned __int128)M0 * c0;
        unsigned __int128 p1 = (unsigned __int128)M1 * c2;
        uint64_t n0 = (uint64_t)(p1 >> 64) ^ c1 ^ k0;
        uint64_t n1 = (uint64_t)p1;
        uint64_t n2 = (uint64_t)(p0 >> 64) ^ c3 ^ k1;
        uint64_t n3 = (uint64_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

int oracle_dropout_keep(uint64_t seed, uint64_t offset, int64_t i, float p)
{
    /* a block serves eight elements: element i takes the 16-bit half
     * (i mod 2: 0 the low half, 1 the high half) of word (i mod 8) / 2 of the
     * block at counter (0, 0, lo(g), hi(g)), g = offset + floor(i / 8), key
     * (lo, hi) of seed */
    uint64_t g = offset + (uint64_t)i / 8u;
    uint32_t ctr[4] = {0u, 0u, (uint32_t)g, (uint32_t)(g >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    uint32_t word = w[(i % 8) / 2];
    uint32_t half = (i % 2) ? (word >> 16) : (word & 0xFFFFu);
    /* u = the half as a fraction in [0, 1): exact in fp32 */
    float u = (float)half * 0x1p-16f;
    return u >= p;
}

void oracle_dropout_mask(uint64_t seed, uint64_t offset, int64_t start, int64_t n, float p,
                         uint8_t *keep)
{
    for (int64_t k = 0; k < n; ++k)
        keep[k] = (uint8_t)oracle_dropout_keep(seed, offset, start + k, p);
}

/* ------------------------------------------------------------------------ */
/* o4: LayerNorm family                                                     */
/* [P3] §4.3 (mean, var = sum((x - mean)^2)/cols, (x - mean)/sqrt(var + eps) */
/* * gamma + beta); [P2] §2.1 (LayerNorm -> ReLU fused) and §2.2-2.3         */
/* (residual + LayerNorm, then GeLU)                                         */
/* ------------------------------------------------------------------------ */

static double o4_act(double n, int act)
{
    if (act == 1)
        return n > 0.0 ? n : 0.0;      /* relu, every value not > 0 to +0 */
    if (act == 2)
        return oracle_gelu_tanh(n);
    return n;
}

/* The optional extras of the LayerNorm family: dropout on the activation
 * (p = 0: none) and the per-row statistics written out (NULL: not written). */
struct o4_extras {
    float p;
    uint64_t seed, offset;
    double *mean_out, *rstd_out;
};

static void o4_rows(const void *x, const void *r, const void *w, const void *b,
                    o3_load_fn load, void *out, void *h_out, int bf16, int64_t rows,
                    int64_t hidden, float eps, int act, const struct o4_extras *ex)
{
    for (int64_t i = 0; i < rows; ++i) {
        int64_t base = i * hidden;
        double sum = 0.0;
        for (int64_t j = 0; j < hidden; ++j) {
            float v = load(x, base + j);
            if (r)
                v = v + load(r, base + j);
            sum += (double)v;
        }
        double mean = sum / (double)hidden;
        double sq = 0.0;
        for (int64_t j = 0; j < hidden; ++j) {
            float v = load(x, base + j);
            if (r)
                v = v + load(r, base + j);
            double d = (double)v - mean;
            sq += d * d;
        }
        double rstd = 1.0 / sqrt(sq / (double)hidden + (double)eps);
        if (ex->mean_out)
            ex->mean_out[i] = mean;
        if (ex->rstd_out)
            ex->rstd_out[i] = rstd;
        for (int64_t j = 0; j < hidden; ++j) {
            float v = load(x, base + j);
            if (r)
                v = v + load(r, base + j);
            if (h_out) {
                if (bf16)
                    ((uint16_t *)h_out)[base + j] = oracle_bf16_from_double((double)v);
                else
                    ((float *)h_out)[base + j] = v;
            }
            double n = ((double)v - mean) * rstd * (double)load(w, j) + (double)load(b, j);
            double g = o4_act(n, act);
            if (ex->p > 0.0f) {
                /* dropout: a kept element is scaled by 1 / (1 - p); a dropped
                 * one is the product g * 0 (a signed zero, as the scaled
                 * mask product of eager dropout gives) */
                if (oracle_dropout_keep(ex->seed, ex->offset, base + j, ex->p))
                    g = g / (1.0 - (double)ex->p);
                else
                    g = g * 0.0;
            }
            if (bf16)
                ((uint16_t *)out)[base + j] = oracle_bf16_from_double(g);
            else
                ((float *)out)[base + j] = (float)g;
        }
    }
}

void oracle_layernorm_act_f32(const float *x, const float *r, const float *w,
                              const float *b, float *out, float *h_out, int64_t rows,
                              int64_t hidden, float eps, int act)
{
    struct o4_extras none = {0.0f, 0, 0, NULL, NULL};
    o4_rows(x, r, w, b, load_f32, out, h_out, 0, rows, hidden, eps, act, &none);
}

void oracle_layernorm_act_bf16(const uint16_t *x, const uint16_t *r, const uint16_t *w,
                               const uint16_t *b, uint16_t *out, uint16_t *h_out,
                               int64_t rows, int64_t hidden, float eps, int act)
{
    struct o4_extras none = {0.0f, 0, 0, NULL, NULL};
    o4_rows(x, r, w, b, load_bf16, out, h_out, 1, rows, hidden, eps, act, &none);
}

void oracle_layernorm_act_ex_f32(const float *x, const float *r, const float *w,
                                 const float *b, float *out, float *h_out, double *mean_out,
                                 double *rstd_out, int64_t rows, int64_t hidden, float eps,
                                 int act, float p, uint64_t seed, uint64_t offset)
{
    struct o4_extras ex = {p, seed, offset, mean_out, rstd_out};
    o4_rows(x, r, w, b, load_f32, out, h_out, 0, rows, hidden, eps, act, &ex);
}

void oracle_layernorm_act_ex_bf16(const uint16_t *x, const uint16_t *r, const uint16_t *w,
                                  const uint16_t *b, uint16_t *out, uint16_t *h_out,
                                  double *mean_out, double *rstd_out, int64_t rows,
                                  int64_t hidden, float eps, int act, float p, uint64_t seed,
                                  uint64_t offset)
{
    struct o4_extras ex = {p, seed, offset, mean_out, rstd_out};
    o4_rows(x, r, w, b, load_bf16, out, h_out, 1, rows, hidden, eps, act, &ex);
}

/* ------------------------------------------------------------------------ */
/* o5: row softmax                                                          */
/* [P1] §4.1-4.2 and [P2] §3.2: softmax over each score row, normalised by  */
/* the row maximum before exponentiation                                     */
/* ------------------------------------------------------------------------ */

static void o5_rows(const void *x, o3_load_fn load, void *y, int bf16, int64_t rows,
                    int64_t cols)
{
    for (int64_t i = 0; i < rows; ++i) {
        int64_t base = i * cols;
        double m = -INFINITY;
        for (int64_t j = 0; j < cols; ++j) {
            double v = (double)load(x, base + j);
            if (v > m)
                m = v;
        }
        double sum = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            sum += exp((double)load(x, base + j) - m);
        for (int64_t j = 0; j < cols; ++j) {
            double p = exp((double)load(x, base + j) - m) / sum;
            if (bf16)
                ((uint16_t *)y)[base + j] = oracle_bf16_from_double(p);
            else
                ((float *)y)[base + j] = (float)p;
        }
    }
}

void oracle_row_softmax_f32(const float *x, float *y, int64_t rows, int64_t cols)
{
    o5_rows(x, load_f32, y, 0, rows, cols);
}

void oracle_row_softmax_bf16(const uint16_t *x, uint16_t *y, int64_t rows, int64_t cols)
{
    o5_rows(x, load_bf16, y, 1, rows, cols);
}

/* o5 on attention scores ([P1] §4.1: the score matrix is scaled before the
 * softmax; §4.2: a causal mask keeps each query from the keys after it):
 * v = x * scale, one fp32 multiply; with causal masking element j of row i is
 * masked when j > (i mod period) + offset (row i is query i mod period of its
 * head; offset aligns the diagonal), and masked elements take no part: the
 * softmax runs in double over the row's unmasked elements, masked outputs
 * are 0. */
static float o5m_value(const void *x, o3_load_fn load, int64_t k, float scale)
{
    float v = load(x, k) * scale;
    return v;
}

static void o5m_rows(const void *x, o3_load_fn load, void *y, int bf16, int64_t rows,
                     int64_t cols, float scale, int causal, int64_t period, int64_t offset)
{
    for (int64_t i = 0; i < rows; ++i) {
        int64_t base = i * cols;
        int64_t end = cols;                     /* elements [0, end) are unmasked */
        if (causal) {
            int64_t last = i % period + offset; /* the last key query i may see */
            if (last + 1 < end)
                end = last + 1;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < end; ++j) {
            double v = (double)o5m_value(x, load, base + j, scale);
            if (v > m)
                m = v;
        }
        double sum = 0.0;
        for (int64_t j = 0; j < end; ++j)
            sum += exp((double)o5m_value(x, load, base + j, scale) - m);
        for (int64_t j = 0; j < cols; ++j) {
            double p = 0.0;
            if (j < end)
                p = exp((double)o5m_value(x, load, base + j, scale) - m) / sum;
            if (bf16)
                ((uint16_t *)y)[base + j] = oracle_bf16_from_double(p);
            else
                ((float *)y)[base + j] = (float)p;
        }
    }
}

void oracle_scale_mask_softmax_f32(const float *x, float *y, int64_t rows, int64_t cols,
                                   float scale, int causal, int64_t period, int64_t offset)
{
    o5m_rows(x, load_f32, y, 0, rows, cols, scale, causal, period, offset);
}

void oracle_scale_mask_softmax_bf16(const uint16_t *x, uint16_t *y, int64_t rows, int64_t cols,
                                    float scale, int causal, int64_t period, int64_t offset)
{
    o5m_rows(x, load_bf16, y, 1, rows, cols, scale, causal, period, offset);
}
