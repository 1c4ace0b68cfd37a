// api.cu -- the C ABI (include/memory_bound.h): argument checks, per-device
// state, dispatch to the kernels, status reporting.
#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"
#include "memory_bound.h"

namespace mb {

namespace {

// Device-side failure flags (one word per device; each device that loads the
// library gets its own copy of this variable).
__device__ unsigned g_dev_err = 0;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int smem_optin = 0;
    int smem_per_sm = 0;
    unsigned *dev_err = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
RowTuning g_tuning{MB_ROW_AUTO, 0, 0, 0};
bool g_pdl = true;
PointwiseTuning g_pw_tuning{0, 0};
thread_local int g_last_cuda_error = 0;

mb_status device_ctx(cudaStream_t stream, LaunchCtx *ctx) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return MB_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                        dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.smem_per_sm,
                                        cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
                cudaSuccess ||
            (e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.dev_err), g_dev_err)) !=
                cudaSuccess)
            return cuda_fail(e);
        d.ready = true;
    }
    *ctx = LaunchCtx{stream, dev, d.sm_count, d.smem_optin, d.smem_per_sm, d.dev_err, g_pdl,
                     g_tuning, g_pw_tuning};
    return MB_OK;
}

inline uintptr_t addr(const void *p) { return reinterpret_cast<uintptr_t>(p); }

// [a, a + na) and [b, b + nb) share a byte.
inline bool overlaps(const void *a, int64_t na, const void *b, int64_t nb) {
    if (na <= 0 || nb <= 0) return false;
    return addr(a) < addr(b) + (uintptr_t)nb && addr(b) < addr(a) + (uintptr_t)na;
}

inline bool aligned_to(const void *p, uintptr_t a) { return (addr(p) & (a - 1)) == 0; }

inline int elem_size(mb_dtype d) { return d == MB_BF16 ? 2 : 4; }

bool valid_dtype(mb_dtype d) { return d == MB_F32 || d == MB_BF16; }

// Alignment class of a row-chain call (the row engines' `aligned`): 1 when
// every pointer is 16-byte aligned; 2 when every row tensor (the row inputs
// and outputs, NULLs skipped) starts at the same offset within 16 bytes and
// the per-column vectors are anywhere; 0 otherwise.
int align_class(std::initializer_list<const void *> row_tensors,
                std::initializer_list<const void *> col_vectors) {
    bool all16 = true, same = true;
    int phase = -1;
    for (const void *p : row_tensors) {
        if (!p) continue;
        const int ph = (int)(addr(p) & 15u);
        all16 = all16 && ph == 0;
        if (phase < 0) phase = ph;
        same = same && ph == phase;
    }
    for (const void *p : col_vectors) all16 = all16 && aligned_to(p, 16);
    return all16 ? 1 : (same ? 2 : 0);
}

// Row-length check shared by the row chains.
mb_status check_rows(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 1 || cols > MB_MAX_COLS) return MB_ERR_SHAPE;
    // rows * cols elements must be addressable
    if (rows > INT64_MAX / cols / 4) return MB_ERR_SHAPE;
    return MB_OK;
}

}  // namespace

cudaError_t launch_kernel(const LaunchCtx &ctx, const void *fn, dim3 grid, dim3 block,
                          void **args, size_t smem, int cluster) {
    if (!ctx.pdl && cluster <= 1) return cudaLaunchKernel(fn, grid, block, args, smem, ctx.stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (ctx.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

mb_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return MB_ERR_CUDA;
}

bool device_resident(const void *p) {
    // The query fails for pointers the runtime does not know, and clearing
    // that failure must not clear an error the calling thread already had
    // pending: with one pending, the pointer is taken as not device memory
    // (the plain-load paths serve any memory) and is not queried.
    if (cudaPeekAtLastError() != cudaSuccess) return false;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();           // an unknown pointer is not an error here
        return false;
    }
    return at.type == cudaMemoryTypeDevice;
}

}  // namespace mb

using namespace mb;

extern "C" {

mb_status fused_add_relu_scale(const void *x, const void *b1, const void *b2, void *y,
                               int64_t n, float scale, mb_dtype dtype, cudaStream_t stream) {
    if (!valid_dtype(dtype)) return MB_ERR_DTYPE;
    if (n < 0 || n > INT64_MAX / 8) return MB_ERR_SHAPE;
    if (!std::isfinite(scale)) return MB_ERR_VALUE;
    if (n == 0) return MB_OK;
    if (!x || !b1 || !b2 || !y) return MB_ERR_NULL;
    const int es = elem_size(dtype);
    for (const void *p : {x, b1, b2, static_cast<const void *>(y)})
        if (!aligned_to(p, es)) return MB_ERR_ALIGN;
    const int64_t bytes = n * es;
    if (overlaps(y, bytes, x, bytes) || overlaps(y, bytes, b1, bytes) ||
        overlaps(y, bytes, b2, bytes))
        return MB_ERR_OVERLAP;
    // Vector path when all four pointers sit at the same offset within 16
    // bytes: a scalar head brings them to a 16-byte boundary together.
    const uintptr_t m = addr(x) & 15;
    const bool vec = (addr(b1) & 15) == m && (addr(b2) & 15) == m && (addr(y) & 15) == m;
    int64_t head = vec ? (int64_t)((16 - m) & 15) / es : 0;
    if (head > n) head = n;
    LaunchCtx ctx;
    mb_status st = device_ctx(stream, &ctx);
    if (st != MB_OK) return st;
    return add_relu_scale_run(ctx, ctx.pw, dtype, x, b1, b2, y, n, scale, vec, (int)head);
}

mb_status fused_add_relu_scale_bcast(const void *x, const void *b1, const void *b2, void *y,
                                     int64_t rows, int64_t cols, int b1_per_col,
                                     int b2_per_col, float scale, mb_dtype dtype,
                                     cudaStream_t stream) {
    if (!valid_dtype(dtype)) return MB_ERR_DTYPE;
    if (rows < 0 || cols < 1 || cols > INT32_MAX || rows > INT64_MAX / 8 / cols)
        return MB_ERR_SHAPE;
    if ((b1_per_col != 0 && b1_per_col != 1) || (b2_per_col != 0 && b2_per_col != 1))
        return MB_ERR_VALUE;
    if (!std::isfinite(scale)) return MB_ERR_VALUE;
    if (rows == 0) return MB_OK;
    if (!x || !b1 || !b2 || !y) return MB_ERR_NULL;
    const int es = elem_size(dtype);
    for (const void *p : {x, b1, b2, static_cast<const void *>(y)})
        if (!aligned_to(p, es)) return MB_ERR_ALIGN;
    const int64_t big = rows * cols * es, small = cols * es;
    if (overlaps(y, big, x, big) || overlaps(y, big, b1, b1_per_col ? small : big) ||
        overlaps(y, big, b2, b2_per_col ? small : big))
        return MB_ERR_OVERLAP;
    if (!b1_per_col && !b2_per_col)       // no broadcast: the plain chain
        return fused_add_relu_scale(x, b1, b2, y, rows * cols, scale, dtype, stream);
    bool vec = cols % (16 / es) == 0;
    for (const void *p : {x, b1, b2, static_cast<const void *>(y)})
        vec = vec && aligned_to(p, 16);
    LaunchCtx ctx;
    mb_status st = device_ctx(stream, &ctx);
    if (st != MB_OK) return st;
    return add_relu_scale_bcast_run(ctx, dtype, x, b1, b2, y, rows, cols, b1_per_col != 0,
                                    b2_per_col != 0, scale, vec);
}

mb_status fused_residual_layernorm_gelu(const void *x, const void *r, const void *w,
                                        const void *b, void *out, int64_t rows,
                                        int64_t hidden, float eps, mb_dtype dtype,
                                        cudaStream_t stream) {
    if (!valid_dtype(dtype)) return MB_ERR_DTYPE;
    mb_status st = check_rows(rows, hidden);
    if (st != MB_OK) return st;
    if (!std::isfinite(eps) || eps < 0.0f) return MB_ERR_VALUE;
    if (rows == 0) return MB_OK;
    if (!x || !r || !w || !b || !out) return MB_ERR_NULL;
    const int es = elem_size(dtype);
    for (const void *p : {x, r, w, b, static_cast<const void *>(out)})
        if (!aligned_to(p, es)) return MB_ERR_ALIGN;
    const int64_t big = rows * hidden * es, small = hidden * es;
    if (overlaps(out, big, x, big) || overlaps(out, big, r, big) ||
        overlaps(out, big, w, small) || overlaps(out, big, b, small))
        return MB_ERR_OVERLAP;
    const int aligned = align_class({x, r, out}, {w, b});
    LaunchCtx ctx;
    if ((st = device_ctx(stream, &ctx)) != MB_OK) return st;
    RowTuning tun = ctx.tuning;
    if (dtype == MB_F32)
        return ln_gelu_rows_f32(ctx, tun, x, r, w, b, out, rows, (int)hidden, eps, aligned,
                                nullptr, true);
    return ln_gelu_rows_bf16(ctx, tun, x, r, w, b, out, rows, (int)hidden, eps, aligned,
                             nullptr, true);
}

mb_status fused_bias_relu_branch_mean_epilogue(const float *x, const float *bias,
                                               const float *gamma, const float *beta,
                                               float *y, int64_t rows, int64_t cols,
                                               float x_scale, float branch_scale,
                                               cudaStream_t stream) {
    mb_status st = check_rows(rows, cols);
    if (st != MB_OK) return st;
    if (!std::isfinite(x_scale) || !std::isfinite(branch_scale)) return MB_ERR_VALUE;
    if (rows == 0) return MB_OK;
    if (!x || !bias || !gamma || !beta || !y) return MB_ERR_NULL;
    for (const void *p : {(const void *)x, (const void *)bias, (const void *)gamma,
                          (const void *)beta, (const void *)y})
        if (!aligned_to(p, 4)) return MB_ERR_ALIGN;
    const int64_t big = rows * cols * 4, small = cols * 4;
    if (overlaps(y, big, x, big) || overlaps(y, big, bias, small) ||
        overlaps(y, big, gamma, small) || overlaps(y, big, beta, small))
        return MB_ERR_OVERLAP;
    const int aligned = align_class({x, y}, {bias, gamma, beta});
    LaunchCtx ctx;
    if ((st = device_ctx(stream, &ctx)) != MB_OK) return st;
    return inductor_rows_f32(ctx, ctx.tuning, x, bias, gamma, beta, y, rows, (int)cols, x_scale,
                             branch_scale, aligned, nullptr, true);
}

mb_status fused_bias_relu_branch_mean_epilogue_bf16(const void *x, const void *bias,
                                                    const void *gamma, const void *beta,
                                                    void *y, int64_t rows, int64_t cols,
                                                    float x_scale, float branch_scale,
                                                    cudaStream_t stream) {
    mb_status st = check_rows(rows, cols);
    if (st != MB_OK) return st;
    if (!std::isfinite(x_scale) || !std::isfinite(branch_scale)) return MB_ERR_VALUE;
    if (rows == 0) return MB_OK;
    if (!x || !bias || !gamma || !beta || !y) return MB_ERR_NULL;
    for (const void *p : {x, bias, gamma, beta, static_cast<const void *>(y)})
        if (!aligned_to(p, 2)) return MB_ERR_ALIGN;
    const int64_t big = rows * cols * 2, small = cols * 2;
    if (overlaps(y, big, x, big) || overlaps(y, big, bias, small) ||
        overlaps(y, big, gamma, small) || overlaps(y, big, beta, small))
        return MB_ERR_OVERLAP;
    const int aligned = align_class({x, y}, {bias, gamma, beta});
    LaunchCtx ctx;
    if ((st = device_ctx(stream, &ctx)) != MB_OK) return st;
    return inductor_rows_bf16(ctx, ctx.tuning, x, bias, gamma, beta, y, rows, (int)cols, x_scale,
                              branch_scale, aligned, nullptr, true);
}

mb_status fused_layernorm_act(const void *x, const void *r, const void *w, const void *b,
                              void *out, void *h_out, int64_t rows, int64_t hidden, float eps,
                              mb_activation act, mb_dtype dtype, cudaStream_t stream) {
    return fused_layernorm_act_ex(x, r, w, b, out, h_out, nullptr, nullptr, rows, hidden, eps,
                                  act, 0.0f, 0, 0, dtype, stream);
}

mb_status fused_layernorm_act_ex(const void *x, const void *r, const void *w, const void *b,
                                 void *out, void *h_out, float *mean_out, float *rstd_out,
                                 int64_t rows, int64_t hidden, float eps, mb_activation act,
                                 float p, uint64_t seed, uint64_t offset, mb_dtype dtype,
                                 cudaStream_t stream) {
    if (!valid_dtype(dtype)) return MB_ERR_DTYPE;
    mb_status st = check_rows(rows, hidden);
    if (st != MB_OK) return st;
    if (!std::isfinite(eps) || eps < 0.0f) return MB_ERR_VALUE;
    if (act != MB_ACT_NONE && act != MB_ACT_RELU && act != MB_ACT_GELU_TANH) return MB_ERR_VALUE;
    if (!(p >= 0.0f && p < 1.0f)) return MB_ERR_VALUE;     // NaN fails too
    if (rows == 0) return MB_OK;
    if (!x || !w || !b || !out) return MB_ERR_NULL;
    const int es = elem_size(dtype);
    for (const void *q : {x, r, w, b, static_cast<const void *>(out),
                          static_cast<const void *>(h_out)})
        if (q && !aligned_to(q, es)) return MB_ERR_ALIGN;
    for (const void *q : {static_cast<const void *>(mean_out),
                          static_cast<const void *>(rstd_out)})
        if (q && !aligned_to(q, 4)) return MB_ERR_ALIGN;
    const int64_t big = rows * hidden * es, small = hidden * es, stat = rows * 4;
    // every output (out, h_out, mean_out, rstd_out) against every input and
    // against the other outputs
    const void *outs[4] = {out, h_out, mean_out, rstd_out};
    const int64_t out_bytes[4] = {big, big, stat, stat};
    for (int i = 0; i < 4; ++i) {
        const void *o = outs[i];
        const int64_t n = out_bytes[i];
        if (!o) continue;
        if (overlaps(o, n, x, big) || (r && overlaps(o, n, r, big)) ||
            overlaps(o, n, w, small) || overlaps(o, n, b, small))
            return MB_ERR_OVERLAP;
        for (int j = i + 1; j < 4; ++j)
            if (outs[j] && overlaps(o, n, outs[j], out_bytes[j])) return MB_ERR_OVERLAP;
    }
    const int aligned = align_class({x, r, out, h_out}, {w, b});
    LaunchCtx ctx;
    if ((st = device_ctx(stream, &ctx)) != MB_OK) return st;
    LnExtras ex;
    ex.mean = mean_out;
    ex.rstd = rstd_out;
    ex.p = p;
    ex.seed = seed;
    ex.offset = offset;
    const bool drop = p > 0.0f;
    auto fn = dtype == MB_F32 ? (drop ? lnact_drop_rows_f32 : lnact_rows_f32)
                              : (drop ? lnact_drop_rows_bf16 : lnact_rows_bf16);
    return fn(ctx, ctx.tuning, r != nullptr, x, r, w, b, out, h_out, rows, (int)hidden, eps,
              (int)act, ex, aligned, nullptr, true);
}

mb_status fused_row_softmax(const void *x, void *y, int64_t rows, int64_t cols, mb_dtype dtype,
                            cudaStream_t stream) {
    if (!valid_dtype(dtype)) return MB_ERR_DTYPE;
    mb_status st = check_rows(rows, cols);
    if (st != MB_OK) return st;
    if (rows == 0) return MB_OK;
    if (!x || !y) return MB_ERR_NULL;
    const int es = elem_size(dtype);
    if (!aligned_to(x, es) || !aligned_to(y, es)) return MB_ERR_ALIGN;
    const int64_t big = rows * cols * es;
    if (overlaps(y, big, x, big)) return MB_ERR_OVERLAP;
    const int aligned = align_class({x, y}, {});
    LaunchCtx ctx;
    if ((st = device_ctx(stream, &ctx)) != MB_OK) return st;
    return softmax_rows(ctx, ctx.tuning, dtype, x, y, rows, (int)cols, aligned, nullptr, true);
}

mb_status fused_scale_mask_softmax(const void *x, void *y, int64_t rows, int64_t cols,
                                   float scale, int causal, int64_t period, int64_t offset,
                                   mb_dtype dtype, cudaStream_t stream) {
    if (!valid_dtype(dtype)) return MB_ERR_DTYPE;
    mb_status st = check_rows(rows, cols);
    if (st != MB_OK) return st;
    if (!std::isfinite(scale) || (causal != 0 && causal != 1)) return MB_ERR_VALUE;
    if (causal && (period < 1 || offset < 0)) return MB_ERR_VALUE;
    if (rows == 0) return MB_OK;
    if (!x || !y) return MB_ERR_NULL;
    const int es = elem_size(dtype);
    if (!aligned_to(x, es) || !aligned_to(y, es)) return MB_ERR_ALIGN;
    const int64_t big = rows * cols * es;
    if (overlaps(y, big, x, big)) return MB_ERR_OVERLAP;
    const int aligned = align_class({x, y}, {});
    LaunchCtx ctx;
    if ((st = device_ctx(stream, &ctx)) != MB_OK) return st;
    return softmax_mask_rows(ctx, ctx.tuning, dtype, x, y, rows, (int)cols, scale, causal != 0,
                             causal ? period : 1, causal ? offset : 0, aligned, nullptr, true);
}

const char *mb_status_string(mb_status s) {
    switch (s) {
        case MB_OK: return "ok";
        case MB_ERR_NULL: return "a required pointer is NULL";
        case MB_ERR_SHAPE: return "invalid or unsupported size";
        case MB_ERR_DTYPE: return "unsupported dtype";
        case MB_ERR_OVERLAP: return "output overlaps an input";
        case MB_ERR_ALIGN: return "pointer not aligned to its element size";
        case MB_ERR_VALUE: return "invalid scalar argument";
        case MB_ERR_CUDA: return "CUDA runtime error";
        case MB_ERR_DEVICE: return "device-side failure recorded";
    }
    return "unknown status";
}

int mb_abi_version(void) { return MB_ABI_VERSION; }

int mb_last_cuda_error(void) { return g_last_cuda_error; }

mb_status mb_device_error(uint32_t *flags) {
    if (!flags) return MB_ERR_NULL;
    LaunchCtx ctx;
    mb_status st = device_ctx(0, &ctx);
    if (st != MB_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned v = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_dev_err, sizeof v)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemcpyToSymbol(g_dev_err, &zero, sizeof zero)) != cudaSuccess)
        return cuda_fail(e);
    *flags = v;
    return v ? MB_ERR_DEVICE : MB_OK;
}

mb_status mb_set_row_path(mb_row_path path, int ctas_per_sm, int stages,
                          int vec_per_thread) {
    if (path < MB_ROW_AUTO || path > MB_ROW_CLUSTER || ctas_per_sm < 0 || stages < 0 ||
        vec_per_thread < 0)
        return MB_ERR_VALUE;
    std::lock_guard<std::mutex> lock(g_mu);
    g_tuning = RowTuning{(int)path, ctas_per_sm, stages, vec_per_thread};
    return MB_OK;
}

mb_status mb_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream) {
    if (limit_us < 1 || limit_us > 1000000) return MB_ERR_VALUE;
    LaunchCtx ctx;
    mb_status st = device_ctx(stream, &ctx);
    if (st != MB_OK) return st;
    return selftest_wait_timeout(ctx, limit_us);
}

mb_status mb_selftest_exchange_timeout(uint32_t limit_us, cudaStream_t stream) {
    if (limit_us < 1 || limit_us > 1000000) return MB_ERR_VALUE;
    LaunchCtx ctx;
    mb_status st = device_ctx(stream, &ctx);
    if (st != MB_OK) return st;
    return selftest_exchange_timeout(ctx, limit_us);
}

mb_status mb_set_launch_overlap(int enable) {
    if (enable != 0 && enable != 1) return MB_ERR_VALUE;
    std::lock_guard<std::mutex> lock(g_mu);
    g_pdl = enable != 0;
    return MB_OK;
}

mb_status mb_set_pointwise_shape(int blocks_per_sm, int unroll) {
    if (blocks_per_sm < 0 || !(unroll == 0 || unroll == 1 || unroll == 2 || unroll == 4 ||
                               unroll == 8))
        return MB_ERR_VALUE;
    std::lock_guard<std::mutex> lock(g_mu);
    g_pw_tuning = PointwiseTuning{blocks_per_sm, unroll};
    return MB_OK;
}

mb_status mb_row_plan(int chain, mb_dtype dtype, int64_t rows, int64_t cols, int aligned,
                      int32_t out[7]) {
    if (!out) return MB_ERR_NULL;
    if (chain < 0 || chain > 8 || aligned < 0 || aligned > 2) return MB_ERR_VALUE;
    if (!valid_dtype(dtype)) return MB_ERR_DTYPE;
    mb_status st = check_rows(rows, cols);
    if (st != MB_OK) return st;
    LaunchCtx ctx;
    if ((st = device_ctx(0, &ctx)) != MB_OK) return st;
    RowPlan p;
    const int al = aligned;
    if (chain == 1 && dtype == MB_F32)
        st = inductor_rows_f32(ctx, ctx.tuning, nullptr, nullptr, nullptr, nullptr, nullptr, rows,
                               (int)cols, 1.0f, 1.0f, al, &p, false);
    else if (chain == 1)
        st = inductor_rows_bf16(ctx, ctx.tuning, nullptr, nullptr, nullptr, nullptr, nullptr, rows,
                                (int)cols, 1.0f, 1.0f, al, &p, false);
    else if (chain == 2 || chain == 3 || chain == 7) {
        RowTuning t = ctx.tuning;
        if (chain == 7) t.outs = 2;            // with the residual-stream output
        st = (dtype == MB_F32 ? lnact_rows_f32 : lnact_rows_bf16)(
            ctx, t, chain != 3, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, rows,
            (int)cols, 0.0f, 0, LnExtras{}, al, &p, false);
    }
    else if (chain == 5 || chain == 6)
        st = (dtype == MB_F32 ? lnact_drop_rows_f32 : lnact_drop_rows_bf16)(
            ctx, ctx.tuning, chain == 5, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, rows,
            (int)cols, 0.0f, 0, LnExtras{}, al, &p, false);
    else if (chain == 4)
        st = softmax_rows(ctx, ctx.tuning, dtype, nullptr, nullptr, rows, (int)cols, al, &p, false);
    else if (chain == 8)
        st = softmax_mask_rows(ctx, ctx.tuning, dtype, nullptr, nullptr, rows, (int)cols, 1.0f,
                               true, cols, 0, al, &p, false);
    else if (dtype == MB_F32)
        st = ln_gelu_rows_f32(ctx, ctx.tuning, nullptr, nullptr, nullptr, nullptr, nullptr, rows,
                              (int)cols, 0.0f, al, &p, false);
    else
        st = ln_gelu_rows_bf16(ctx, ctx.tuning, nullptr, nullptr, nullptr, nullptr, nullptr, rows,
                               (int)cols, 0.0f, al, &p, false);
    if (st != MB_OK) return st;
    out[0] = p.path; out[1] = p.threads; out[2] = p.ctas; out[3] = p.vpt;
    out[4] = p.vec; out[5] = p.stages; out[6] = p.smem;
    return MB_OK;
}

}  // extern "C"
