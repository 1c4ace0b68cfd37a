// rows.cuh -- row engines for the reduce-plus-pointwise chains.
//
// A chain C supplies, per row of `cols` elements:
//   pre   (per element)   the pointwise prologue, giving v from the row inputs
//   mean  = sum(v) / cols (always), and with C::kTwoPass
//   rstd  = C::rstd(sum((v - mean)^2), cols, args)   (second pass over v)
//   post  (per element)   the epilogue from v, mean, rstd
// The row is read from device memory once and held in registers (v) between
// the passes; the output is written once.
//
// Engines:
//   rows_warp_kernel  one warp per row (rows of <= 256 vectors): loads straight
//                     into registers, shuffle reductions only, no barriers.
//   rows_cta_kernel   one CTA per row, persistent over rows (row b, b + G, ...):
//     DIRECT  vector loads into registers;
//     STAGED  one elected thread streams whole rows into a ring of shared
//             memory stages with bulk async copies (cp.async.bulk completing
//             on an mbarrier per stage) up to `nstage` rows ahead; the ring
//             slot of row i is refilled with row i + nstage as soon as the
//             first reduction barrier shows that every thread has copied row
//             i into registers.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace mb {

constexpr int kCtaMaxThreads = 1024;
constexpr int kWarpBlock = 256;
constexpr int kHdrBytes = 1024;   // reduction buffers, abort flags, mbarriers
constexpr int kMaxStages = 16;

// ---------------------------------------------------------------------------
// one warp per row
// ---------------------------------------------------------------------------
template <class C, int VPL, int VEC>
__global__ void __launch_bounds__(kWarpBlock)
rows_warp_kernel(const typename C::Args a, int64_t rows, int cols, int, unsigned *) {
    using T = typename C::T;
    constexpr int NIN = C::kInputs;
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nvec = cols / VEC;
    for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows;
         row += nw) {
        const int64_t base = row * cols;
        float v[VPL][VEC];
        float lsum = 0.0f;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int vi = lane + 32 * k;
            if (vi < nvec) {
                Frag<T, VEC> in[NIN];
#pragma unroll
                for (int i = 0; i < NIN; ++i) in[i].load_stream(a.in[i] + base + vi * VEC);
                C::template pre<VEC>(in, a, vi * VEC, v[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) lsum += v[k][e];
            }
        }
        const float mean = warp_sum(lsum) / (float)cols;
        float rstd = 0.0f;
        if constexpr (C::kTwoPass) {
            float lm2 = 0.0f;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                if (lane + 32 * k < nvec) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float d = v[k][e] - mean;
                        lm2 = fmaf(d, d, lm2);
                    }
                }
            }
            rstd = C::rstd(warp_sum(lm2), cols, a);
        }
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int vi = lane + 32 * k;
            if (vi < nvec) {
                Frag<T, VEC> o;
                C::template post<VEC>(v[k], mean, rstd, a, vi * VEC, o.f);
                o.store_stream(a.out + base + vi * VEC);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// one CTA per row, persistent; DIRECT or STAGED (bulk-async shared ring)
// ---------------------------------------------------------------------------
template <class C, int VPT, int VEC, bool STAGED>
__global__ void __launch_bounds__(kCtaMaxThreads)
rows_cta_kernel(const typename C::Args a, int64_t rows, int cols, int nstage, unsigned *err) {
    using T = typename C::T;
    constexpr int NIN = C::kInputs;
    extern __shared__ __align__(1024) unsigned char smem[];
    float *red = reinterpret_cast<float *>(smem);                  // [2][32]
    volatile int *abort_flag = reinterpret_cast<int *>(smem + 256); // [2]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 512);     // [kMaxStages]
    unsigned char *ring = smem + kHdrBytes;

    const int tid = threadIdx.x;
    const int nvec = cols / VEC;
    const int64_t G = gridDim.x;
    const int64_t first = blockIdx.x;
    const int64_t nlocal = (rows - first + G - 1) / G;   // host: G <= rows
    const uint32_t row_bytes = (uint32_t)cols * (uint32_t)sizeof(T);
    const uint32_t stage_bytes = (uint32_t)NIN * row_bytes;

    if (tid == 0) {
        abort_flag[0] = 0;
        abort_flag[1] = 0;
        if constexpr (STAGED) {
            for (int s = 0; s < nstage; ++s) mbar_init(smem_addr(&bars[s]), 1);
            fence_mbar_init();
        }
    }
    __syncthreads();

    // Refill ring slot s with local row li (one elected thread).
    auto issue = [&](int s, int64_t li) {
        const int64_t row = first + li * G;
        const uint32_t bar = smem_addr(&bars[s]);
        mbar_arrive_expect_tx(bar, stage_bytes);
#pragma unroll
        for (int i = 0; i < NIN; ++i)
            bulk_g2s(smem_addr(ring + (size_t)s * stage_bytes + (size_t)i * row_bytes),
                     a.in[i] + row * cols, row_bytes, bar);
    };
    if constexpr (STAGED) {
        if (tid == 0) {
            const int64_t n0 = nlocal < nstage ? nlocal : nstage;
            for (int s = 0; s < (int)n0; ++s) issue(s, s);
        }
    }

    int rb = 0;
    int64_t li = 0;
    for (; li < nlocal; ++li) {
        const int64_t row = first + li * G;
        const int64_t base = row * cols;
        const int s = STAGED ? (int)(li % nstage) : 0;
        const T *stage = reinterpret_cast<const T *>(ring + (size_t)s * stage_bytes);
        if constexpr (STAGED) {
            const uint32_t parity = (uint32_t)((li / nstage) & 1);
            if (!mbar_wait_bounded(smem_addr(&bars[s]), parity)) abort_flag[li & 1] = 1;
        }

        float v[VPT][VEC];
        float lsum = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vi = tid + k * blockDim.x;
            if (vi < nvec) {
                Frag<T, VEC> in[NIN];
#pragma unroll
                for (int i = 0; i < NIN; ++i) {
                    if constexpr (STAGED) in[i].load_shared(stage + (size_t)i * cols + vi * VEC);
                    else in[i].load_stream(a.in[i] + base + vi * VEC);
                }
                C::template pre<VEC>(in, a, vi * VEC, v[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) lsum += v[k][e];
            }
        }
        // Barrier inside: after it every thread has its row slice in registers.
        const float sum = block_sum(lsum, red + 32 * rb);
        rb ^= 1;
        if constexpr (STAGED) {
            if (abort_flag[li & 1]) break;
            if (tid == 0 && li + nstage < nlocal) issue(s, li + nstage);
        }
        const float mean = sum / (float)cols;
        float rstd = 0.0f;
        if constexpr (C::kTwoPass) {
            float lm2 = 0.0f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                if (tid + k * (int)blockDim.x < nvec) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float d = v[k][e] - mean;
                        lm2 = fmaf(d, d, lm2);
                    }
                }
            }
            rstd = C::rstd(block_sum(lm2, red + 32 * rb), cols, a);
            rb ^= 1;
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vi = tid + k * blockDim.x;
            if (vi < nvec) {
                Frag<T, VEC> o;
                C::template post<VEC>(v[k], mean, rstd, a, vi * VEC, o.f);
                o.store_stream(a.out + base + vi * VEC);
            }
        }
    }
    if constexpr (STAGED) {
        // Only after a timed-out wait: record it, and wait (bounded) for this
        // CTA's copies still in flight before its shared memory goes away.
        if (li < nlocal && tid == 0) {
            atomicOr(err, kDevErrWaitTimeout);
            for (int64_t lj = li; lj < nlocal && lj < li + nstage; ++lj)
                (void)mbar_wait_bounded(smem_addr(&bars[lj % nstage]), (uint32_t)((lj / nstage) & 1));
        }
    }
}

// ---------------------------------------------------------------------------
// host-side planning and launch
// ---------------------------------------------------------------------------

inline int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }
inline int round_up32(int v) { return (v + 31) & ~31; }

// Raises a kernel's dynamic shared memory limit to the device's opt-in
// maximum (needed above 48 KB, before occupancy queries and launches).
inline cudaError_t allow_smem(const void *fn, const LaunchCtx &ctx, int bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ctx.smem_optin);
}

template <class C> struct RowEngine {
    using T = typename C::T;
    static constexpr int kVecN = Elem<T>::kVec;

    // Kernel table.  Index: vectors per thread slot as a power of two.
    static const void *warp_fn(int vpl, bool vec) {
        if (vec) {
            switch (vpl) {
                case 1: return (const void *)rows_warp_kernel<C, 1, kVecN>;
                case 2: return (const void *)rows_warp_kernel<C, 2, kVecN>;
                case 4: return (const void *)rows_warp_kernel<C, 4, kVecN>;
                case 8: return (const void *)rows_warp_kernel<C, 8, kVecN>;
            }
        } else {
            switch (vpl) {
                case 1: return (const void *)rows_warp_kernel<C, 1, 1>;
                case 2: return (const void *)rows_warp_kernel<C, 2, 1>;
                case 4: return (const void *)rows_warp_kernel<C, 4, 1>;
                case 8: return (const void *)rows_warp_kernel<C, 8, 1>;
            }
        }
        return nullptr;
    }
    // Vector slots per thread allowed on the CTA engine: VPT * VEC <= 32.
    static int max_vpt(bool vec) { return vec ? 32 / kVecN : 32; }
    static const void *cta_fn(int vpt, bool vec, bool staged) {
        if (vec) {
            if (staged) {
                switch (vpt) {
                    case 1: return (const void *)rows_cta_kernel<C, 1, kVecN, true>;
                    case 2: return (const void *)rows_cta_kernel<C, 2, kVecN, true>;
                    case 4: return (const void *)rows_cta_kernel<C, 4, kVecN, true>;
                    case 8: if constexpr (kVecN == 4) return (const void *)rows_cta_kernel<C, 8, kVecN, true>;
                            break;
                }
            } else {
                switch (vpt) {
                    case 1: return (const void *)rows_cta_kernel<C, 1, kVecN, false>;
                    case 2: return (const void *)rows_cta_kernel<C, 2, kVecN, false>;
                    case 4: return (const void *)rows_cta_kernel<C, 4, kVecN, false>;
                    case 8: if constexpr (kVecN == 4) return (const void *)rows_cta_kernel<C, 8, kVecN, false>;
                            break;
                }
            }
        } else if (!staged) {
            switch (vpt) {
                case 1: return (const void *)rows_cta_kernel<C, 1, 1, false>;
                case 2: return (const void *)rows_cta_kernel<C, 2, 1, false>;
                case 4: return (const void *)rows_cta_kernel<C, 4, 1, false>;
                case 8: return (const void *)rows_cta_kernel<C, 8, 1, false>;
                case 16: return (const void *)rows_cta_kernel<C, 16, 1, false>;
                case 32: return (const void *)rows_cta_kernel<C, 32, 1, false>;
            }
        }
        return nullptr;
    }

    static mb_status plan(const LaunchCtx &ctx, const RowTuning &tun, int64_t rows, int cols,
                          bool aligned, RowPlan *p, const void **fn) {
        const bool vec = aligned && (cols % kVecN) == 0;
        const int VEC = vec ? kVecN : 1;
        const int nvec = cols / VEC;
        const bool warp_ok = nvec <= 32 * 8;
        const int64_t stage_bytes = (int64_t)C::kInputs * cols * (int64_t)sizeof(T);

        int path = tun.path;
        if (path == MB_ROW_WARP && !warp_ok) path = MB_ROW_AUTO;
        if (path == MB_ROW_STAGED && !vec) path = MB_ROW_AUTO;
        if (path == MB_ROW_AUTO) path = warp_ok ? MB_ROW_WARP : (vec ? MB_ROW_STAGED : MB_ROW_DIRECT);

        p->vec = VEC;
        if (path == MB_ROW_WARP) {
            int vpl = 1;
            while (vpl * 32 < nvec) vpl *= 2;
            *fn = warp_fn(vpl, vec);
            int occ = 0;
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, *fn, kWarpBlock, 0);
            if (e != cudaSuccess) return cuda_fail(e);
            if (tun.ctas_per_sm > 0 && tun.ctas_per_sm < occ) occ = tun.ctas_per_sm;
            if (occ < 1) occ = 1;
            const int64_t want = (rows + kWarpBlock / 32 - 1) / (kWarpBlock / 32);
            const int64_t cap = (int64_t)occ * ctx.sm_count;
            p->path = path; p->threads = kWarpBlock; p->vpt = vpl; p->stages = 0; p->smem = 0;
            p->ctas = (int)(want < cap ? want : cap);
            return MB_OK;
        }

        // CTA engine: smallest VPT giving <= 512 threads, else <= 1024.
        int vpt = 0;
        for (int cand = 1; cand <= max_vpt(vec); cand *= 2)
            if (ceil_div(nvec, cand) <= 512) { vpt = cand; break; }
        if (!vpt)
            for (int cand = 1; cand <= max_vpt(vec); cand *= 2)
                if (ceil_div(nvec, cand) <= kCtaMaxThreads) { vpt = cand; break; }
        if (!vpt) return MB_ERR_SHAPE;
        const int threads = round_up32(ceil_div(nvec, vpt));

        int stages = 0, smem = kHdrBytes;
        int target = tun.ctas_per_sm > 0 ? tun.ctas_per_sm : (threads <= 512 ? 2 : 1);
        if (path == MB_ROW_STAGED) {
            for (; target >= 1; --target) {
                const int per_cta = ctx.smem_per_sm / target - 1024;   // 1 KB reserved per CTA
                const int budget = (per_cta < ctx.smem_optin ? per_cta : ctx.smem_optin) - kHdrBytes;
                int64_t n = budget / stage_bytes;
                if (n > kMaxStages) n = kMaxStages;
                if (tun.stages > 0 && tun.stages < n) n = tun.stages;
                if (n >= 2 || (tun.stages == 1 && n >= 1)) { stages = (int)n; break; }
            }
            if (!stages) path = MB_ROW_DIRECT;
            else smem = kHdrBytes + (int)(stages * stage_bytes);
        }
        *fn = cta_fn(vpt, vec, path == MB_ROW_STAGED);
        if (!*fn) return MB_ERR_SHAPE;
        cudaError_t e = allow_smem(*fn, ctx, smem);
        if (e != cudaSuccess) return cuda_fail(e);
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, *fn, threads, smem);
        if (e != cudaSuccess) return cuda_fail(e);
        if (occ < 1) occ = 1;
        if (path == MB_ROW_STAGED && occ > target) occ = target;
        if (path == MB_ROW_DIRECT && tun.ctas_per_sm > 0 && tun.ctas_per_sm < occ)
            occ = tun.ctas_per_sm;
        const int64_t cap = (int64_t)occ * ctx.sm_count;
        p->path = path; p->threads = threads; p->vpt = vpt; p->stages = stages; p->smem = smem;
        p->ctas = (int)(rows < cap ? rows : cap);
        return MB_OK;
    }

    static mb_status run(const LaunchCtx &ctx, const RowTuning &tun, const typename C::Args &a,
                         int64_t rows, int cols, bool aligned, RowPlan *plan_out, bool launch) {
        RowPlan p;
        const void *fn = nullptr;
        mb_status st = plan(ctx, tun, rows, cols, aligned, &p, &fn);
        if (st != MB_OK) return st;
        if (plan_out) *plan_out = p;
        if (!launch || rows == 0) return MB_OK;
        typename C::Args args = a;
        int64_t rows_arg = rows;
        int cols_arg = cols;
        int stages_arg = p.stages > 0 ? p.stages : 1;
        unsigned *err = ctx.dev_err;
        void *kargs[] = {&args, &rows_arg, &cols_arg, &stages_arg, &err};
        cudaError_t e = cudaLaunchKernel(fn, dim3(p.ctas), dim3(p.threads), kargs, p.smem,
                                         ctx.stream);
        if (e != cudaSuccess) return cuda_fail(e);
        return MB_OK;
    }
};

}  // namespace mb
