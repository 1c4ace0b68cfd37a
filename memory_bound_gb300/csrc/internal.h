// internal.h -- host-side declarations shared by the library's translation
// units (not part of the public ABI; see include/memory_bound.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "memory_bound.h"

namespace mb {

// Launch overlap pays for calls whose launch latency is a visible share of
// their run time; above this many bytes moved it is noise (measured on GB300:
// +-1%), so those launches keep plain stream order.
constexpr int64_t kOverlapMaxBytes = 128ll << 20;

// Process-wide row-chain override (mb_set_row_path).
struct RowTuning {
    int path;              // mb_row_path
    int ctas_per_sm;       // 0 = automatic
    int stages;            // 0 = automatic
    int vpt;               // vector slots per thread, 0 = automatic
    // per-call planning inputs (set by the row engine, not by the override)
    int no_bulk = 0;       // 1: some input that the planned copies would read is
                           // not device memory, so no asynchronous copies into
                           // shared memory are planned (the STAGED path, the
                           // cluster ring, the shifted kernel's per-column copies)
    int outs = 1;          // full-size outputs written per row (2 with the
                           // LayerNorm family's residual-stream output)
    int read_pct = 100;    // share of each row's input elements read, on
                           // average over the rows (percent, 1..100)
};

// Process-wide pointwise override (mb_set_pointwise_shape).
struct PointwiseTuning {
    int blocks_per_sm;     // 0 = as many as fit
    int unroll;            // 16-byte fragments per input in flight per thread; 0 = 4
};

// What a launcher needs to know about the current device and stream, and
// the process-wide overrides as they stood when the call began.
struct LaunchCtx {
    cudaStream_t stream;
    int device;
    int sm_count;
    int smem_optin;        // max dynamic shared memory per block (opt-in)
    int smem_per_sm;       // shared memory per multiprocessor
    unsigned *dev_err;     // device-side failure flags of this device
    bool pdl;              // launch with programmatic stream serialisation
    RowTuning tuning;      // the row-chain override, read under the state lock
    PointwiseTuning pw;    // the pointwise override, read under the state lock
};

// cudaLaunchKernel, or cudaLaunchKernelEx with programmatic stream
// serialisation when ctx.pdl (the kernels wait for their predecessor).
cudaError_t launch_kernel(const LaunchCtx &ctx, const void *fn, dim3 grid, dim3 block,
                          void **args, size_t smem, int cluster = 1);

// The launch a row chain uses (mb_row_plan reports it).
struct RowPlan {
    int path = 0, threads = 0, ctas = 0, vpt = 0, vec = 0, stages = 0, smem = 0;
    int slice = 0;     // cluster path: vectors of the row each CTA holds
    int shift = 0;     // rows off the 16-byte grid (shifted vectors): 1; on the one-CTA
                       // path 2 with the per-column values copied to shared memory, 3
                       // with the copies and the staged ring
    int ring = 0;      // cluster path: staging ring depth (0: direct loads)
    int64_t cap = 0;   // CTAs (warp/CTA paths, at 256 threads for warp) or clusters resident at once
    int64_t cap1 = 0;  // shift 2, 3: CTAs of the same launch in the plain shifted form
                       // resident at once
};

// Chains implemented in their own translation units.  `launch == false`
// only fills `plan`.
mb_status add_relu_scale_run(const LaunchCtx &ctx, const PointwiseTuning &tun, mb_dtype dtype,
                             const void *x, const void *b1, const void *b2, void *y, int64_t n,
                             float scale, bool vec, int head);
// rows x cols with b1 / b2 per column where flagged; vec: 16-byte fragments
// (every pointer 16-byte aligned and cols a multiple of the fragment length).
mb_status add_relu_scale_bcast_run(const LaunchCtx &ctx, mb_dtype dtype, const void *x,
                                   const void *b1, const void *b2, void *y, int64_t rows,
                                   int64_t cols, bool b1_per_col, bool b2_per_col, float scale,
                                   bool vec);

mb_status ln_gelu_rows_f32(const LaunchCtx &ctx, const RowTuning &tun, const void *x,
                           const void *r, const void *w, const void *b, void *out,
                           int64_t rows, int cols, float eps, int aligned,
                           RowPlan *plan, bool launch);
mb_status ln_gelu_rows_bf16(const LaunchCtx &ctx, const RowTuning &tun, const void *x,
                            const void *r, const void *w, const void *b, void *out,
                            int64_t rows, int cols, float eps, int aligned,
                            RowPlan *plan, bool launch);
mb_status inductor_rows_f32(const LaunchCtx &ctx, const RowTuning &tun, const float *x,
                            const float *bias, const float *gamma, const float *beta,
                            float *y, int64_t rows, int cols, float x_scale,
                            float branch_scale, int aligned, RowPlan *plan, bool launch);

mb_status inductor_rows_bf16(const LaunchCtx &ctx, const RowTuning &tun, const void *x,
                             const void *bias, const void *gamma, const void *beta, void *y,
                             int64_t rows, int cols, float x_scale, float branch_scale,
                             int aligned, RowPlan *plan, bool launch);
// Optional extras of the LayerNorm family: per-row statistics out (NULL: not
// written) and dropout with probability p (0: none) keyed by (seed, offset).
struct LnExtras {
    float *mean = nullptr;
    float *rstd = nullptr;
    float p = 0.0f;
    uint64_t seed = 0;
    uint64_t offset = 0;
};

// LayerNorm family launches: fp32 / bf16 I/O, without dropout (lnact_rows_*)
// and with it (lnact_drop_rows_*, p > 0).
#define MB_LNACT_DECL(name)                                                              \
    mb_status name(const LaunchCtx &ctx, const RowTuning &tun, bool residual, const void *x, \
                   const void *r, const void *w, const void *b, void *out, void *h,          \
                   int64_t rows, int cols, float eps, int act, const LnExtras &ex,           \
                   int aligned, RowPlan *plan, bool launch)
MB_LNACT_DECL(lnact_rows_f32);
MB_LNACT_DECL(lnact_rows_bf16);
MB_LNACT_DECL(lnact_drop_rows_f32);
MB_LNACT_DECL(lnact_drop_rows_bf16);
#undef MB_LNACT_DECL
mb_status softmax_mask_rows(const LaunchCtx &ctx, const RowTuning &tun, mb_dtype dtype,
                            const void *x, void *y, int64_t rows, int cols, float scale,
                            bool causal, int64_t period, int64_t offset, int aligned,
                            RowPlan *plan, bool launch);
mb_status softmax_rows(const LaunchCtx &ctx, const RowTuning &tun, mb_dtype dtype,
                       const void *x, void *y, int64_t rows, int cols, int aligned,
                       RowPlan *plan, bool launch);

mb_status selftest_wait_timeout(const LaunchCtx &ctx, uint32_t limit_us);
mb_status selftest_exchange_timeout(const LaunchCtx &ctx, uint32_t limit_us);

// Records a CUDA error for mb_last_cuda_error and returns MB_ERR_CUDA.
mb_status cuda_fail(cudaError_t e);

// True when p lies in device memory (cudaMalloc, stream-ordered or virtual
// memory allocations); false for pinned or other host memory, managed memory
// and pointers CUDA does not know.  Only device memory is bulk-copied.
bool device_resident(const void *p);

}  // namespace mb
