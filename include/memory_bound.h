/*
 * memory_bound.h -- C ABI of the fused memory-bound chain library
 * (libmemory_bound.so, CUDA for sm_103a).
 *
 * Three vertically fused chains, each one kernel launch that reads its inputs
 * from device memory once and writes its output once:
 *
 *   fused_add_relu_scale                  y = relu(x + b1) * scale + b2
 *   fused_bias_relu_branch_mean_epilogue  the TorchInductor example chain
 *   fused_residual_layernorm_gelu         GeLU_tanh(LayerNorm(x + r) * w + b)
 *
 * with the broadcast form of the first, fused_add_relu_scale_bcast
 * (per-column b1 / b2), and, built on the same row engines,
 * fused_layernorm_act (LayerNorm with an optional residual, residual-stream
 * output and activation) and its extended form fused_layernorm_act_ex
 * (dropout, per-row statistics), fused_row_softmax, its scaled and causally
 * masked form fused_scale_mask_softmax and the bf16 variant of the
 * TorchInductor chain.
 *
 * Sources (the pages these chains come from):
 *   [P1] "PyTorch operator fusion in practice", www.0539edu.com/news/5489619
 *   [P2] "Operator fusion and kernel optimisation: from CUDA Graph to
 *        FlashAttention", plumephp.com/ai-kernel-fusion-optimization
 *   [P3] "Kernel fusion", course chapter 4, www.5688vip.com
 *   [P4] "TorchInductor Pipeline and operator fusion", blog.kkkzoz.top
 *
 * Conventions shared by every entry point:
 *
 *   Pointers    Device pointers, or any pointer the current device can
 *               dereference at the same address: page-locked host memory
 *               (cudaHostAlloc / cudaMallocHost, mapped into the device's
 *               address space) included.  The kernels then read and write
 *               that memory directly over the host link ("zero copy"); row
 *               inputs that are not device memory never go through the
 *               bulk-async staged path (each call checks them with
 *               cudaPointerGetAttributes when that path is planned), so
 *               host rows take a plain-load path.  The caller owns every
 *               buffer, outputs included: the library never allocates,
 *               frees or copies buffers and never synchronises the stream.
 *   Layout      Contiguous, row-major.  Per-column vectors (length cols /
 *               hidden) are broadcast over all rows (a stride-0 row view).
 *   dtype       MB_F32 (IEEE binary32) or MB_BF16 (bfloat16, raw 16-bit
 *               patterns).  All tensors of one call share the dtype;
 *               arithmetic is fp32 and bf16 results are rounded to nearest,
 *               ties to even.
 *   Alignment   Every pointer must be aligned to its element size, else
 *               MB_ERR_ALIGN.  Pointers that are 16-byte aligned (and rows
 *               whose byte length is a multiple of 16) take the vectorised
 *               paths.  Row chains whose rows are off that grid (a row
 *               length that is not a whole number of 16-byte vectors, or
 *               row tensors starting off a 16-byte boundary) still take
 *               16-byte row accesses when all row tensors of the call (row
 *               inputs and outputs) start at the same offset within 16
 *               bytes and a row holds one CTA's worth or less: each row is
 *               then read as a short head, whole vectors and a short tail.
 *               Anything else runs on a scalar path.
 *   Aliasing    The output may not overlap any input (MB_ERR_OVERLAP).
 *               Inputs may overlap one another.
 *   Sizes       Zero rows / zero elements is a no-op returning MB_OK without
 *               touching the GPU.  Row lengths are 1 .. MB_MAX_COLS.
 *   Stream      Work is enqueued on `stream` (0 = the legacy default stream)
 *               on the current device.  The call is asynchronous; no host
 *               synchronisation, allocation or host-device copy happens, so
 *               calls may be captured into a CUDA graph.
 *   Errors      Argument errors are found on the host before anything is
 *               launched, and the call returns without side effects.
 *               A failed launch returns MB_ERR_CUDA (see mb_last_cuda_error).
 *               Faults during execution surface at the caller's next
 *               synchronisation, as for any CUDA kernel.  The staged row paths
 *               and the cluster path wait on shared-memory barriers with a
 *               time limit; if a wait ever ran out, the kernel stops early and
 *               records it in a device flag that mb_device_error() reports.
 *   Threads     Entry points may be called from several host threads.
 *               mb_set_row_path changes process-wide state and should not
 *               race with calls.
 */
#ifndef MEMORY_BOUND_H
#define MEMORY_BOUND_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MB_ABI_VERSION 1

/* Longest row (cols / hidden) the row chains accept.  Rows longer than one
 * CTA can hold (32768 elements) are spread over a thread-block cluster of up
 * to 16 CTAs. */
#define MB_MAX_COLS 524288

typedef enum mb_status {
    MB_OK = 0,
    MB_ERR_NULL = 1,      /* a pointer that must be read or written is NULL     */
    MB_ERR_SHAPE = 2,     /* negative size, zero row length, or above a limit   */
    MB_ERR_DTYPE = 3,     /* dtype code not supported by this entry point      */
    MB_ERR_OVERLAP = 4,   /* the output range overlaps an input range          */
    MB_ERR_ALIGN = 5,     /* a pointer is not aligned to its element size      */
    MB_ERR_VALUE = 6,     /* a scalar argument is NaN/inf, or eps < 0          */
    MB_ERR_CUDA = 7,      /* the CUDA runtime reported an error                */
    MB_ERR_DEVICE = 8     /* a kernel recorded a device-side failure           */
} mb_status;

typedef enum mb_dtype {
    MB_F32 = 0,
    MB_BF16 = 1
} mb_dtype;

/* ------------------------------------------------------------------------ */
/* Fused chains                                                             */
/* ------------------------------------------------------------------------ */

/*
 * y[i] = relu(x[i] + b1[i]) * scale + b2[i],   0 <= i < n.
 *
 * [P1] §1.1 (the chain and its four eager kernels) and §3.2 (the fused
 * float4 kernel, with relu written fmaxf(v, 0)).  fp32: the four operations
 * are rounded one at a time in that order (no fused multiply-add), so the
 * result equals the eager fp32 sequence bit for bit.  relu maps every value
 * that is not > 0 (including -0 and NaN) to +0.  bf16: inputs are widened
 * exactly, the same fp32 sequence runs, and y is rounded once to bf16.
 *
 *   x, b1, b2  n elements each (inputs)         y  n elements (output)
 *   n >= 0     scale finite                     dtype MB_F32 or MB_BF16
 */
mb_status fused_add_relu_scale(const void *x, const void *b1, const void *b2,
                               void *y, int64_t n, float scale, mb_dtype dtype,
                               cudaStream_t stream);

/*
 * TorchInductor example chain, row by row over a rows x cols fp32 matrix:
 *   t = x * x_scale + bias[j];  a = relu(t);  p = a * a;  q = a * branch_scale;
 *   s = p + q;  m[i] = mean_j s[i, j];  y = (s - m[i]) * gamma[j] + beta[j]
 *
 * [P4] the example model at the top of the post (x_scale = 1.1,
 * branch_scale = 0.1), Figure 1, §6.4 (the mean is a row sum divided by the
 * row length) and §08 (one persistent-reduction kernel: x read once, the row
 * sum kept on chip, y written once).  The pointwise steps are rounded one at
 * a time as fp32 ops; the row sum is an fp32 tree sum; relu as above.
 *
 *   x      rows x cols (input)          bias, gamma, beta   cols each (input)
 *   y      rows x cols (output)         rows >= 0, 1 <= cols <= MB_MAX_COLS
 *   x_scale, branch_scale finite
 */
mb_status fused_bias_relu_branch_mean_epilogue(const float *x, const float *bias,
                                               const float *gamma,
                                               const float *beta, float *y,
                                               int64_t rows, int64_t cols,
                                               float x_scale, float branch_scale,
                                               cudaStream_t stream);

/*
 * The pointwise chain over rows x cols with b1 and / or b2 given per column:
 *   y[i, j] = relu(x[i, j] + B1(i, j)) * scale + B2(i, j),
 *   Bk(i, j) = bk[j] when bk_per_col (a length-cols vector broadcast over the
 *   rows, as a bias is), else bk[i * cols + j].
 * [P1] §3.1's chain with bias-like operands; the same four fp32 steps per
 * element, each rounded on its own, so fp32 results are bit-identical to the
 * eager ops with broadcasting (bf16: inputs widened exactly, y rounded once).
 *
 *   x, y        rows x cols
 *   b1, b2      cols values when the flag is 1, rows x cols when it is 0
 *   b1_per_col, b2_per_col   0 or 1, else MB_ERR_VALUE; with both 0 this is
 *               fused_add_relu_scale over rows * cols elements
 *   rows >= 0 (0: no-op), 1 <= cols <= INT32_MAX, else MB_ERR_SHAPE
 *   y may not overlap x, b1 or b2 (MB_ERR_OVERLAP).
 */
mb_status fused_add_relu_scale_bcast(const void *x, const void *b1, const void *b2, void *y,
                                     int64_t rows, int64_t cols, int b1_per_col,
                                     int b2_per_col, float scale, mb_dtype dtype,
                                     cudaStream_t stream);

/*
 * out = GeLU_tanh(LayerNorm(x + r) * w + b), row by row over rows x hidden:
 *   v = x + r;  mean = sum(v)/H;  var = sum((v - mean)^2)/H  (biased);
 *   rstd = 1/sqrt(var + eps);  n = (v - mean) * rstd * w[j] + b[j];
 *   out = 0.5 n (1 + tanh(sqrt(2/pi) (n + 0.044715 n^3)))
 *
 * [P2] §2.2-2.3 (the residual + LayerNorm + GeLU fused kernel; the affine
 * step is applied before the GeLU, as its code does) and [P3] §4.3 (LayerNorm:
 * mean, two-pass variance, (v - mean)/sqrt(var + eps) * gamma + beta).
 * v is the fp32 sum of the (widened) inputs; statistics are fp32 tree sums
 * over the row held on chip (two passes); the output is rounded once to the
 * I/O dtype.
 *
 *   x, r   rows x hidden (input)        w, b   hidden each (input)
 *   out    rows x hidden (output)       rows >= 0, 1 <= hidden <= MB_MAX_COLS
 *   eps    finite, >= 0                 dtype  MB_F32 or MB_BF16 (all tensors)
 */
mb_status fused_residual_layernorm_gelu(const void *x, const void *r,
                                        const void *w, const void *b, void *out,
                                        int64_t rows, int64_t hidden, float eps,
                                        mb_dtype dtype, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Further chains: the LayerNorm family, row softmax, bf16 Inductor chain   */
/* ------------------------------------------------------------------------ */

typedef enum mb_activation {
    MB_ACT_NONE = 0,
    MB_ACT_RELU = 1,        /* every value not > 0 (including -0, NaN) -> +0 */
    MB_ACT_GELU_TANH = 2
} mb_activation;

/*
 * The LayerNorm family, row by row over rows x hidden:
 *   v = x + r  (or v = x when r is NULL);  h_out = v  (when h_out is not NULL);
 *   mean, biased two-pass variance, rstd = 1/sqrt(var + eps);
 *   out = act((v - mean) * rstd * w[j] + b[j])
 *
 * [P3] §4.3 (LayerNorm: mean, two-pass variance, (x - mean)/sqrt(var + eps) *
 * gamma + beta), [P2] §2.1 (LayerNorm -> ReLU in one kernel) and §2.2-2.3
 * (residual + LayerNorm, then GeLU).  h_out is the residual stream a
 * Transformer block carries on: the fp32 sum rounded once to the I/O dtype.
 * Arithmetic as in fused_residual_layernorm_gelu.
 *
 *   x, r   rows x hidden (input; r may be NULL)     w, b  hidden each (input)
 *   out    rows x hidden (output)                    h_out rows x hidden (output, may be NULL)
 *   act    an mb_activation; other codes give MB_ERR_VALUE
 *   out and h_out may not overlap each other or any input.
 */
mb_status fused_layernorm_act(const void *x, const void *r, const void *w, const void *b,
                              void *out, void *h_out, int64_t rows, int64_t hidden,
                              float eps, mb_activation act, mb_dtype dtype,
                              cudaStream_t stream);

/*
 * fused_layernorm_act with its optional extras, in the same single pass:
 *
 *   dropout  [P2] §2.1 fuses LayerNorm -> ReLU -> Dropout (p = 0.1 there)
 *            into one kernel.  With 0 < p < 1 each element of `out` is kept
 *            with probability 1 - p and scaled by 1 / (1 - p) (fp32, rounded
 *            once), or multiplied by 0.  The pages fix no random number
 *            generator; the decision is the counter-based Philox-4x32-10
 *            ("Parallel random numbers: as easy as 1, 2, 3", SC'11), one
 *            16-bit uniform per element: element i = row * hidden + col takes
 *            the half h (i mod 2: low, high) of word (i mod 8) / 2 of the block
 *            at counter (0, 0, lo(g), hi(g)), g = offset + floor(i / 8), under
 *            the key (lo(seed), hi(seed)), and is kept iff h * 2^-16 >= p (so
 *            the drop probability is ceil(p 2^16) / 2^16).  The decisions
 *            depend only on (seed, offset, i, p), never on the launch; a later
 *            call takes fresh ones with offset advanced by
 *            ceil(rows * hidden / 8).  p = 0: no dropout (out is bit-identical
 *            to fused_layernorm_act).  p outside [0, 1) (or NaN) gives
 *            MB_ERR_VALUE.  h_out (the residual stream) is never dropped.
 *   stats    mean_out / rstd_out (fp32, `rows` values each; NULL: not
 *            written) receive each row's mean and 1/sqrt(var + eps), the
 *            statistics the normalisation used (what a LayerNorm backward
 *            pass reads).  4-byte aligned, else MB_ERR_ALIGN.
 *
 * No output (out, h_out, mean_out, rstd_out) may overlap an input or another
 * output (MB_ERR_OVERLAP).
 */
mb_status fused_layernorm_act_ex(const void *x, const void *r, const void *w, const void *b,
                                 void *out, void *h_out, float *mean_out, float *rstd_out,
                                 int64_t rows, int64_t hidden, float eps, mb_activation act,
                                 float p, uint64_t seed, uint64_t offset, mb_dtype dtype,
                                 cudaStream_t stream);

/*
 * Row softmax over rows x cols:  y[i, j] = exp(x[i, j] - m_i) / sum_k exp(x[i, k] - m_i),
 * m_i the row maximum.  [P1] §4.1-4.2 and [P2] §3.2 (the softmax of a score
 * row, normalised by the row maximum; here the row is held on chip, so it is
 * read once).  fp32 arithmetic; exponentials on the SFU (2^(d log2 e)).
 *
 *   x  rows x cols (input)    y  rows x cols (output)    1 <= cols <= MB_MAX_COLS
 */
mb_status fused_row_softmax(const void *x, void *y, int64_t rows, int64_t cols,
                            mb_dtype dtype, cudaStream_t stream);

/*
 * Softmax of attention-score rows, scaled and optionally causally masked:
 *   v[i, j] = x[i, j] * scale (one fp32 multiply; the caller passes 1/sqrt(d));
 *   key j of row i is masked when causal and j > (i mod period) + offset;
 *   y[i, j] = exp(v[i, j] - m_i) / sum_k exp(v[i, k] - m_i) over the unmasked
 *   keys (m_i their maximum), and y = 0 where masked.
 * [P1] §4.1 (the score matrix divided by a scale before the softmax, rows of
 * batch x heads x seq_len queries) and §4.2 (a causal mask that keeps each
 * query from the keys after it).  Rows are (batch, head, query) flattened
 * with `period` queries per head; offset >= 0 aligns the diagonal (seq_k -
 * seq_q for bottom-right alignment), so no row is fully masked.  Masked keys
 * take no part whatever their value, and the masked tail of a row is not read
 * on the staged paths.
 *
 *   x, y    rows x cols (input, output)        1 <= cols <= MB_MAX_COLS
 *   scale   finite, else MB_ERR_VALUE
 *   causal  0 or 1; with 1, period >= 1 and offset >= 0, else MB_ERR_VALUE
 */
mb_status fused_scale_mask_softmax(const void *x, void *y, int64_t rows, int64_t cols,
                                   float scale, int causal, int64_t period, int64_t offset,
                                   mb_dtype dtype, cudaStream_t stream);

/*
 * fused_bias_relu_branch_mean_epilogue with bf16 I/O: x, bias, gamma, beta
 * and y are bf16 bit patterns; inputs are widened exactly, the same fp32
 * steps run, and y is rounded once to bf16.
 */
mb_status fused_bias_relu_branch_mean_epilogue_bf16(const void *x, const void *bias,
                                                    const void *gamma, const void *beta,
                                                    void *y, int64_t rows, int64_t cols,
                                                    float x_scale, float branch_scale,
                                                    cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Status, diagnostics and tuning                                           */
/* ------------------------------------------------------------------------ */

/* Static, NUL-terminated description of a status code. */
const char *mb_status_string(mb_status s);

/* MB_ABI_VERSION of the loaded library. */
int mb_abi_version(void);

/* The cudaError_t (as int) behind the last MB_ERR_CUDA returned on the
 * calling host thread; 0 if none. */
int mb_last_cuda_error(void);

/*
 * Reads and clears the device-side failure flags of the current device
 * (bit 0: a staged-row or cluster-exchange barrier wait ran out of time).  Synchronises the
 * device.  *flags receives the bits; returns MB_ERR_DEVICE if any bit was
 * set, MB_OK if none, MB_ERR_NULL / MB_ERR_CUDA on failure.
 */
mb_status mb_device_error(uint32_t *flags);

/*
 * Self-test of the failure path: launches one thread that waits, with a limit
 * of limit_us microseconds (1 .. 1000000), on a shared-memory barrier that
 * nothing completes -- the same bounded wait the staged row kernels use.  The
 * wait runs out, the kernel records bit 0 in the device flags and ends
 * normally, so a following mb_device_error() reports MB_ERR_DEVICE and the
 * context stays usable.  Asynchronous on `stream`.
 */
mb_status mb_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream);

/*
 * Self-test of the cluster exchange's failure path: a cluster of two CTAs
 * exchanges partials as the cluster row kernels do (st.async pushes that
 * complete bytes on each CTA's own mbarrier), except that one push is never
 * sent.  The waiting CTA's bounded wait (limit_us microseconds, 1 .. 1000000)
 * runs out and records bit 0 in the device flags; both CTAs end normally.
 * Asynchronous on `stream`.
 */
mb_status mb_selftest_exchange_timeout(uint32_t limit_us, cudaStream_t stream);

/* Row-chain execution paths (all row chains). */
typedef enum mb_row_path {
    MB_ROW_AUTO = 0,     /* choose by shape and alignment (default)            */
    MB_ROW_WARP = 1,     /* one warp per row, row in registers                */
    MB_ROW_DIRECT = 2,   /* one CTA per row, vector loads into registers      */
    MB_ROW_STAGED = 3,   /* one CTA per row, rows staged into shared memory by
                            bulk async copies in a multi-stage ring            */
    MB_ROW_CLUSTER = 4   /* one thread-block cluster per row: each CTA holds a
                            slice in registers (bf16 rows in vectorised device
                            memory staged by bulk async copies, fp32 rows
                            loaded directly unless a ring depth is asked for;
                            softmax slices of 64 KB or more staged, bf16 ones
                            kept in shared memory), statistics combined
                            through distributed shared memory (automatic above
                            32768 elements)                                    */
} mb_row_path;

/*
 * Process-wide override of the row-chain path and launch shape, for tuning
 * and testing.  ctas_per_sm (CTAs resident per SM; the staging ring depth on
 * the cluster path), stages (ring depth of the staged path; CTAs per row,
 * 2..16, on the cluster path) and vec_per_thread (vector slots each thread
 * holds per row on the CTA and cluster paths; a power of two) of 0 mean
 * "choose automatically"; a
 * value that cannot serve a shape is ignored.  A forced path that cannot
 * serve a shape (MB_ROW_WARP beyond 256 vectors per row, MB_ROW_STAGED on
 * rows too long for one stage or off the 16-byte grid without a common
 * offset, one-CTA paths on rows longer than one CTA holds) falls back to the
 * automatic choice.  Rows off the 16-byte grid with a common offset (shifted
 * vectors) take a staged form when the chain has per-column arrays and it
 * fits; MB_ROW_DIRECT keeps them unstaged.  Returns MB_ERR_VALUE on a bad
 * code or a negative count.
 */
mb_status mb_set_row_path(mb_row_path path, int ctas_per_sm, int stages,
                          int vec_per_thread);

/*
 * Launch overlap (default on): calls that move at most 128 MiB are launched
 * with programmatic stream serialisation, so their launch and prologue overlap
 * the tail of the previous kernel in the stream.  Every kernel of this library waits
 * (griddepcontrol.wait) for the previous grid to complete before touching
 * global memory, so results do not change.  enable 0 / 1; else MB_ERR_VALUE.
 */
mb_status mb_set_launch_overlap(int enable);

/*
 * Process-wide override of the pointwise chain's launch shape, for tuning and
 * testing: blocks_per_sm (0 = as many as fit) and unroll, the 16-byte
 * fragments per input each thread keeps in flight (1, 2, 4 or 8; 0 = the
 * default 4).  Returns MB_ERR_VALUE on a negative count or another unroll.
 */
mb_status mb_set_pointwise_shape(int blocks_per_sm, int unroll);

/*
 * The launch the row chains would use for a shape, without launching:
 * out[0] = path (mb_row_path), out[1] = threads per CTA, out[2] = CTAs,
 * out[3] = values per thread slot (vectors per thread), out[4] = vector width
 * in elements, out[5] = ring stages (staged path), CTAs per row (cluster
 * path), else 0,
 * out[6] = dynamic shared memory bytes.  `chain`: 0 residual + LayerNorm +
 * GeLU, 1 the TorchInductor chain, 2 the LayerNorm family with a residual,
 * 3 without, 4 row softmax, 5 and 6 the LayerNorm family with dropout (with
 * a residual, without), 7 the LayerNorm family with a residual that also
 * writes the residual stream h, 8 the scaled softmax under a square causal
 * mask (period = cols, offset 0: row i reads keys 0 .. i mod cols).
 * `aligned`: 1 every pointer is 16-byte aligned; 2 the row tensors start at
 * one common offset within 16 bytes (per-column vectors anywhere); 0 neither;
 * else MB_ERR_VALUE.  Rows planned on shifted vectors report path
 * MB_ROW_DIRECT, or MB_ROW_STAGED with their ring depth in out[5] (or, longer
 * than a CTA holds, MB_ROW_CLUSTER), with the vector width in out[4] while
 * cols is not a multiple of it; out[6] then
 * includes the shared-memory copy of the chain's per-column arrays where one
 * is planned (launches of several rows a CTA) and the ring.  Queries the
 * current device (SM count, shared memory).
 */
mb_status mb_row_plan(int chain, mb_dtype dtype, int64_t rows, int64_t cols,
                      int aligned, int32_t out[7]);

#ifdef __cplusplus
}
#endif

#endif /* MEMORY_BOUND_H */
