// pointwise.cu -- y = relu(x + b1) * scale + b2, one streaming pass.
//
// "PyTorch operator fusion in practice" (0539edu.com) §1.1 and §3.2: the four
// eager kernels (add, relu, mul, add) become one kernel that reads x, b1, b2
// once and writes y once, with 16-byte vector accesses.  Here the grid is
// sized to the SM count, each CTA owns an equal contiguous share, and each
// thread keeps UNROLL independent 16-byte loads per input in flight; the unaligned head and the ragged tail are done
// in-kernel (no padding by the caller).
#include "common.cuh"
#include "internal.h"

namespace mb {
namespace {

constexpr int kThreads = 256;

// Elements [0, head) and [head + nvec*VEC, n) are done one by one by the
// first threads of block 0; [head, head + nvec*VEC) by 16-byte fragments.
// Block b owns the contiguous fragment range [b*chunk, (b+1)*chunk): every
// block gets the same share, so no block runs a partial extra wave.
template <typename T, int VEC, int UNROLL>
__global__ void __launch_bounds__(kThreads)
add_relu_scale_kernel(const T *__restrict__ x, const T *__restrict__ b1,
                      const T *__restrict__ b2, T *__restrict__ y, int64_t n, int head,
                      int64_t nvec, int64_t chunk, float scale) {
    using F = Frag<T, VEC>;
    using F1 = Frag<T, 1>;
    const int64_t body_end = head + nvec * VEC;
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0) {
        const int t = threadIdx.x;
        const int64_t tail = n - body_end;
        int64_t i = -1;
        if (t < head) i = t;
        else if (t - head < tail) i = body_end + (t - head);
        if (i >= 0) {
            F1 fx, f1, f2, fy;
            fx.load_stream(x + i); f1.load_stream(b1 + i); f2.load_stream(b2 + i);
            fy.f[0] = add_relu_scale_1(fx.f[0], f1.f[0], f2.f[0], scale);
            fy.store_stream(y + i);
        }
    }
    const T *xv = x + head, *b1v = b1 + head, *b2v = b2 + head;
    T *yv = y + head;
    const int64_t start = (int64_t)blockIdx.x * chunk;
    const int64_t end = start + chunk < nvec ? start + chunk : nvec;
    for (int64_t base = start + threadIdx.x; base < end; base += (int64_t)kThreads * UNROLL) {
        // All 3 * UNROLL loads are issued before any is used; slots past the
        // block's end re-read its last fragment (in bounds) and are not stored.
        F fx[UNROLL], f1[UNROLL], f2[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            int64_t i = base + (int64_t)u * kThreads;
            i = i < end ? i : end - 1;
            fx[u].load_stream(xv + i * VEC);
            f1[u].load_stream(b1v + i * VEC);
            f2[u].load_stream(b2v + i * VEC);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + (int64_t)u * kThreads;
            if (i < end) {
                F fy;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    fy.f[e] = add_relu_scale_1(fx[u].f[e], f1[u].f[e], f2[u].f[e], scale);
                fy.store_stream(yv + i * VEC);
            }
        }
    }
}

template <typename T, int VEC>
const void *kernel_for(int unroll) {
    switch (unroll) {
        case 1: return (const void *)add_relu_scale_kernel<T, VEC, 1>;
        case 2: return (const void *)add_relu_scale_kernel<T, VEC, 2>;
        case 8: return (const void *)add_relu_scale_kernel<T, VEC, 8>;
        default: return (const void *)add_relu_scale_kernel<T, VEC, 4>;
    }
}

template <typename T>
mb_status launch(const LaunchCtx &ctx, const PointwiseTuning &tun, const void *x,
                 const void *b1, const void *b2, void *y, int64_t n, float scale, bool vec,
                 int head) {
    constexpr int VN = Elem<T>::kVec;
    const int unroll = tun.unroll > 0 ? tun.unroll : 4;
    const void *fn;
    int64_t nvec;
    if (vec) {
        fn = kernel_for<T, VN>(unroll);
        nvec = (n - head) / VN;
    } else {
        fn = kernel_for<T, 1>(unroll);
        head = 0;
        nvec = n;
    }
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kThreads, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    if (tun.blocks_per_sm > 0 && tun.blocks_per_sm < occ) occ = tun.blocks_per_sm;
    if (occ < 1) occ = 1;
    const int64_t tile = (int64_t)kThreads * unroll;
    int64_t grid = (nvec + tile - 1) / tile;
    const int64_t cap = (int64_t)occ * ctx.sm_count;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;   // block 0 also does the head and tail
    // equal shares, whole warps of fragments (512-byte aligned for fp32)
    int64_t chunk = (nvec + grid - 1) / grid;
    chunk = (chunk + 31) & ~(int64_t)31;
    if (chunk < 1) chunk = 1;
    const T *px = static_cast<const T *>(x), *p1 = static_cast<const T *>(b1),
            *p2 = static_cast<const T *>(b2);
    T *py = static_cast<T *>(y);
    void *args[] = {&px, &p1, &p2, &py, &n, &head, &nvec, &chunk, &scale};
    LaunchCtx lctx = ctx;
    lctx.pdl = ctx.pdl && n * (int64_t)sizeof(T) * 4 <= kOverlapMaxBytes;
    e = launch_kernel(lctx, fn, dim3((unsigned)grid), dim3(kThreads), args, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    return MB_OK;
}

}  // namespace

mb_status add_relu_scale_run(const LaunchCtx &ctx, const PointwiseTuning &tun, mb_dtype dtype,
                             const void *x, const void *b1, const void *b2, void *y, int64_t n,
                             float scale, bool vec, int head) {
    if (dtype == MB_F32) return launch<float>(ctx, tun, x, b1, b2, y, n, scale, vec, head);
    return launch<uint16_t>(ctx, tun, x, b1, b2, y, n, scale, vec, head);
}

}  // namespace mb
