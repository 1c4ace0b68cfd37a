// pointwise_bcast.cu -- y = relu(x + b1) * scale + b2 over rows x cols with b1
// and / or b2 given per column: a length-cols vector broadcast over the rows,
// as a bias is ("PyTorch operator fusion in practice" (0539edu.com) §3.1's
// chain with bias-like operands).  The broadcast vectors are small and are
// read through the read-only cache, so HBM sees x, the full operands and y
// once each.
//
// The tensor is walked as one flat range of 16-byte fragments (rows hold a
// whole number of them on the vector path), split into equal contiguous
// shares per CTA as in the plain pointwise kernel; a fragment's column is
// kept incrementally (one 64-bit remainder per thread, then adds), so any
// row length, short or long, keeps every access coalesced.
#include "common.cuh"
#include "internal.h"

namespace mb {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// nvec fragments in all, ncv per row; C1 / C2: b1 / b2 per column.
template <typename T, int VEC, bool C1, bool C2>
__global__ void __launch_bounds__(kThreads)
add_relu_scale_bcast_kernel(const T *__restrict__ x, const T *__restrict__ b1,
                            const T *__restrict__ b2, T *__restrict__ y, int64_t nvec, int ncv,
                            int64_t chunk, float scale) {
    using F = Frag<T, VEC>;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t start = (int64_t)blockIdx.x * chunk;
    const int64_t end = start + chunk < nvec ? start + chunk : nvec;
    const int step1 = kThreads % ncv;                                  // per slot
    const int stepk = (int)(((int64_t)kThreads * kUnroll) % ncv);      // per iteration
    int64_t base = start + threadIdx.x;
    int c0 = (int)(base % ncv);           // column fragment of `base`
    for (; base < end; base += (int64_t)kThreads * kUnroll) {
        // All loads first.  Slots past the share's end re-read its last
        // fragment (in bounds) and are not stored; their column c is that of
        // the unclamped index, which is in [0, ncv) all the same.
        F fx[kUnroll], f1[kUnroll], f2[kUnroll];
        int c = c0;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            int64_t i = base + (int64_t)u * kThreads;
            i = i < end ? i : end - 1;
            fx[u].load_stream(x + i * VEC);
            if constexpr (C1) f1[u].load_cached(b1 + (int64_t)c * VEC);
            else f1[u].load_stream(b1 + i * VEC);
            if constexpr (C2) f2[u].load_cached(b2 + (int64_t)c * VEC);
            else f2[u].load_stream(b2 + i * VEC);
            c += step1;
            if (c >= ncv) c -= ncv;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + (int64_t)u * kThreads;
            if (i < end) {
                F fy;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    fy.f[e] = add_relu_scale_1(fx[u].f[e], f1[u].f[e], f2[u].f[e], scale);
                fy.store_stream(y + i * VEC);
            }
        }
        c0 += stepk;
        if (c0 >= ncv) c0 -= ncv;
    }
}

template <typename T, int VEC>
const void *kernel_for(bool c1, bool c2) {
    if (c1 && c2) return (const void *)add_relu_scale_bcast_kernel<T, VEC, true, true>;
    if (c1) return (const void *)add_relu_scale_bcast_kernel<T, VEC, true, false>;
    if (c2) return (const void *)add_relu_scale_bcast_kernel<T, VEC, false, true>;
    return (const void *)add_relu_scale_bcast_kernel<T, VEC, false, false>;
}

template <typename T>
mb_status launch(const LaunchCtx &ctx, const void *x, const void *b1, const void *b2, void *y,
                 int64_t rows, int64_t cols, bool c1, bool c2, float scale, bool vec) {
    constexpr int VN = Elem<T>::kVec;
    const int v = vec ? VN : 1;
    const void *fn = vec ? kernel_for<T, VN>(c1, c2) : kernel_for<T, 1>(c1, c2);
    int ncv = (int)(cols / v);
    int64_t nvec = rows * (int64_t)ncv;
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kThreads, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    if (occ < 1) occ = 1;
    const int64_t tile = (int64_t)kThreads * kUnroll;
    int64_t grid = (nvec + tile - 1) / tile;
    const int64_t cap = (int64_t)occ * ctx.sm_count;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    int64_t chunk = (nvec + grid - 1) / grid;
    chunk = (chunk + 31) & ~(int64_t)31;
    grid = (nvec + chunk - 1) / chunk;        // no CTA without a share
    const T *px = static_cast<const T *>(x), *p1 = static_cast<const T *>(b1),
            *p2 = static_cast<const T *>(b2);
    T *py = static_cast<T *>(y);
    void *args[] = {&px, &p1, &p2, &py, &nvec, &ncv, &chunk, &scale};
    LaunchCtx lctx = ctx;
    lctx.pdl = ctx.pdl && rows * cols * (int64_t)sizeof(T) * 4 <= kOverlapMaxBytes;
    e = launch_kernel(lctx, fn, dim3((unsigned)grid), dim3(kThreads), args, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    return MB_OK;
}

}  // namespace

mb_status add_relu_scale_bcast_run(const LaunchCtx &ctx, mb_dtype dtype, const void *x,
                                   const void *b1, const void *b2, void *y, int64_t rows,
                                   int64_t cols, bool b1_per_col, bool b2_per_col, float scale,
                                   bool vec) {
    if (dtype == MB_F32)
        return launch<float>(ctx, x, b1, b2, y, rows, cols, b1_per_col, b2_per_col, scale, vec);
    return launch<uint16_t>(ctx, x, b1, b2, y, rows, cols, b1_per_col, b2_per_col, scale, vec);
}

}  // namespace mb
