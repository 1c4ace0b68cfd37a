/*
 * oracle.h -- plain, slow, obviously correct CPU definitions of the three
 * fused memory-bound chains.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this code; only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load it.  It shares no source with the CUDA
 * path.
 *
 * Sources (the four web pages on vertically fused memory-bound chains):
 *   [P1] "PyTorch operator fusion in practice", www.0539edu.com/news/5489619
 *   [P2] "Operator fusion and kernel optimisation: from CUDA Graph to
 *        FlashAttention", plumephp.com/ai-kernel-fusion-optimization
 *   [P3] "Kernel fusion" course chapter 4, www.5688vip.com (AI training
 *        operator performance, chapter 04)
 *   [P4] "TorchInductor Pipeline and operator fusion", blog.kkkzoz.top
 *        (posts/ml-systems/ml-compilers/torchinductor-fusion)
 *
 * Conventions: all arrays are contiguous row-major; bf16 values travel as
 * their raw 16-bit patterns (uint16_t).  Compile with -ffp-contract=off so
 * that every fp32 operation written below is rounded separately.
 */
#ifndef MB_ORACLE_H
#define MB_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- scalar helpers (exported so the tests can pin them directly) ---- */

/* relu as the [P1] §3.2 kernel writes it (fmaxf(v, 0)), with the two cases
 * fmaxf leaves open fixed: NaN -> +0 and -0 -> +0. */
float oracle_relu_f32(float v);

/* GeLU, tanh form, [P2] §2.3: 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))),
 * evaluated in double. */
double oracle_gelu_tanh(double z);

/* Round a double to the nearest bf16, ties to even (one rounding). */
uint16_t oracle_bf16_from_double(double v);
/* Exact widening of a bf16 bit pattern. */
double oracle_bf16_to_double(uint16_t h);

/* ---- o1: pointwise chain y = relu(x + b1) * scale + b2 ([P1] §1.1, §3.1) ---- */

void oracle_add_relu_scale_f32(const float *x, const float *b1, const float *b2,
                               float *y, int64_t n, float scale);
void oracle_add_relu_scale_bf16(const uint16_t *x, const uint16_t *b1,
                                const uint16_t *b2, uint16_t *y, int64_t n,
                                float scale);

/* ---- o1 over rows x cols with b1 and/or b2 per column: a length-cols vector
 * broadcast over the rows when the flag is set, else a full rows x cols
 * tensor; the same four fp32 steps per element (bf16: widened inputs, y
 * rounded once). */
void oracle_add_relu_scale_bcast_f32(const float *x, const float *b1, const float *b2,
                                     float *y, int64_t rows, int64_t cols, int b1_per_col,
                                     int b2_per_col, float scale);
void oracle_add_relu_scale_bcast_bf16(const uint16_t *x, const uint16_t *b1,
                                      const uint16_t *b2, uint16_t *y, int64_t rows,
                                      int64_t cols, int b1_per_col, int b2_per_col, float scale);

/* ---- o2: TorchInductor example chain ([P4] "model", Figure 1, §6.4) ----
 *   t = x*x_scale + bias; a = relu(t); p = a*a; q = a*branch_scale;
 *   s = p + q; m = mean(s, dim=1); y = (s - m)*gamma + beta
 * s_out (rows*cols) and m_out (rows) are optional intermediates (NULL skips). */
void oracle_bias_relu_branch_mean_epilogue(const float *x, const float *bias,
                                           const float *gamma, const float *beta,
                                           float *y, int64_t rows, int64_t cols,
                                           float x_scale, float branch_scale,
                                           float *s_out, float *m_out);

/* ---- o3: residual + LayerNorm + affine + GeLU-tanh ([P2] §2.2-2.3, [P3] §4.3)
 *   v = x + r; mean, biased var over the row; rstd = 1/sqrt(var + eps);
 *   n = (v - mean)*rstd*w + b; out = gelu_tanh(n)
 * mean_out, rstd_out (rows) and xhat_out (rows*hidden, the pre-affine
 * (v - mean)*rstd) are optional intermediates (NULL skips). */
void oracle_residual_layernorm_gelu_f32(const float *x, const float *r,
                                        const float *w, const float *b,
                                        float *out, int64_t rows, int64_t hidden,
                                        float eps, double *mean_out,
                                        double *rstd_out, double *xhat_out);
void oracle_residual_layernorm_gelu_bf16(const uint16_t *x, const uint16_t *r,
                                         const uint16_t *w, const uint16_t *b,
                                         uint16_t *out, int64_t rows,
                                         int64_t hidden, float eps,
                                         double *mean_out, double *rstd_out,
                                         double *xhat_out);

/* ---- o2 with bf16 I/O: inputs widened exactly, the same fp32 steps and
 * double row sum, y rounded once to bf16. */
void oracle_bias_relu_branch_mean_epilogue_bf16(const uint16_t *x, const uint16_t *bias,
                                                const uint16_t *gamma, const uint16_t *beta,
                                                uint16_t *y, int64_t rows, int64_t cols,
                                                float x_scale, float branch_scale);

/* ---- o4: LayerNorm family ([P3] §4.3 LayerNorm; [P2] §2.1-2.3 residual add,
 * LayerNorm -> ReLU, LayerNorm + GeLU):
 *   v = x (+ r when r is not NULL), in fp32;  h_out = v (when not NULL);
 *   out = act((v - mean) * rstd * w + b),  act: 0 none, 1 relu, 2 gelu_tanh.
 * Statistics as in o3 (double, biased two-pass variance, eps inside sqrt). */
void oracle_layernorm_act_f32(const float *x, const float *r, const float *w,
                              const float *b, float *out, float *h_out, int64_t rows,
                              int64_t hidden, float eps, int act);
void oracle_layernorm_act_bf16(const uint16_t *x, const uint16_t *r, const uint16_t *w,
                               const uint16_t *b, uint16_t *out, uint16_t *h_out,
                               int64_t rows, int64_t hidden, float eps, int act);

/* ---- o4 with the optional extras: per-row statistics written out (mean and
 * rstd in double; NULL: not written) and dropout on the activation output
 * ([P2] §2.1 LayerNorm -> ReLU -> Dropout; p = 0: none), the decision of
 * element i (its index in the whole tensor) as in oracle_dropout_keep; kept
 * values become act / (1 - p) (in double, then rounded once), dropped ones
 * act * 0. */
void oracle_layernorm_act_ex_f32(const float *x, const float *r, const float *w,
                                 const float *b, float *out, float *h_out, double *mean_out,
                                 double *rstd_out, int64_t rows, int64_t hidden, float eps,
                                 int act, float p, uint64_t seed, uint64_t offset);
void oracle_layernorm_act_ex_bf16(const uint16_t *x, const uint16_t *r, const uint16_t *w,
                                  const uint16_t *b, uint16_t *out, uint16_t *h_out,
                                  double *mean_out, double *rstd_out, int64_t rows,
                                  int64_t hidden, float eps, int act, float p, uint64_t seed,
                                  uint64_t offset);

/* ---- o6: Philox-4xW-10 ("Parallel random numbers: as easy as 1, 2, 3",
 * SC'11) for W = 32 (the dropout generator) and W = 64 (the same round
 * structure, checkable against numpy's Philox), and the dropout decision:
 *   element i of a call keyed by (seed, offset) takes the 16-bit half h
 *   (i mod 2: low, high) of word (i mod 8) / 2 of Philox-4x32-10 at counter
 *   (0, 0, lo(g), hi(g)), g = offset + floor(i / 8), key (lo(seed),
 *   hi(seed)); u = h * 2^-16; kept iff u >= p. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]);
int oracle_dropout_keep(uint64_t seed, uint64_t offset, int64_t i, float p);
void oracle_dropout_mask(uint64_t seed, uint64_t offset, int64_t start, int64_t n, float p,
                         uint8_t *keep);

/* ---- o5: row softmax ([P1] §4.1-4.2, [P2] §3.2: the softmax of each score
 * row, taken relative to the row maximum):
 *   m = max_j x_j;  e_j = exp(x_j - m);  y_j = e_j / sum_k e_k   (in double) */
void oracle_row_softmax_f32(const float *x, float *y, int64_t rows, int64_t cols);
void oracle_row_softmax_bf16(const uint16_t *x, uint16_t *y, int64_t rows, int64_t cols);

/* ---- o5 on attention scores ([P1] §4.1 scaled scores, §4.2 causal mask):
 *   v = x * scale (one fp32 multiply); causal: element j of row i is masked
 *   when j > (i mod period) + offset; y = softmax over the unmasked elements
 *   (double, as o5), masked outputs 0.  period >= 1, offset >= 0. */
void oracle_scale_mask_softmax_f32(const float *x, float *y, int64_t rows, int64_t cols,
                                   float scale, int causal, int64_t period, int64_t offset);
void oracle_scale_mask_softmax_bf16(const uint16_t *x, uint16_t *y, int64_t rows, int64_t cols,
                                    float scale, int causal, int64_t period, int64_t offset);

#ifdef __cplusplus
}
#endif

#endif /* MB_ORACLE_H */
