// rows.cuh -- row engines for the reduce-plus-pointwise chains.
//
// A chain C supplies, per row of `cols` elements:
//   pre   (per element)   the pointwise prologue, giving v from the row inputs
//                         and the per-column values it needs (PrePC)
//   s1    = C::stat1(R1, cols, args), R1 = sum(v), or max(v) with C::kMaxFirst
//   s2    = C::stat2(R2, cols, args) with C::kTwoPass, where R2 sums the
//           per-slot partials C::p2 forms from v and s1 (p2 may rewrite v)
//   post  (per element)   the epilogue from v, s1, s2, its per-column
//                         values (PostPC) and the index of the slot's first
//                         element in the whole tensor
//   store_stats           one thread per row may write s1 and s2 out
//   early (per slot)      values the epilogue needs that depend only on the
//                         element index (dropout's random bits), drawn while
//                         the row is still in flight and passed to post
// and, with C::kStorePre, store_pre writes the prologue value v out as well
// (the residual-stream output of a residual + LayerNorm block).
// The row is read from device memory once and held in registers (v) between
// the passes; the output is written once.
//
// Engines:
//   rows_warp_kernel  one warp per row (rows of <= 256 vectors): every load of
//                     the row and of its per-column values is issued at once,
//                     shuffle reductions only, no barriers.
//   rows_cta_kernel   one CTA per row, persistent over rows (row b, b + G, ...):
//     DIRECT  vector loads into registers;
//     STAGED  one elected thread streams whole rows into a ring of shared
//             memory stages with bulk async copies (cp.async.bulk completing
//             on an mbarrier per stage) up to `nstage` rows ahead; the ring
//             slot of row i is refilled with row i + nstage as soon as the
//             first reduction barrier shows that every thread has copied row
//             i into registers.
//     (rows_cta_kernel_wide: the scalar forms with many slots per thread,
//     bounded at 512 threads; rows_cta_kernel_capped: the register-capped
//     form a chain may ask for)
//   rows_shift_kernel one CTA per row for rows off the 16-byte grid whose
//                     tensors share one offset within 16 bytes: a short head,
//                     whole 16-byte vectors, a short tail; the per-column
//                     values copied once per CTA into shared memory, aligned
//                     to the CTA's rows (CS).
//   rows_cluster_kernel / rows_cluster_smem_kernel  one thread-block cluster
//                     per row, for rows longer than one CTA holds.
// Several CTAs share an SM, each with its own row in flight, so one CTA's
// loads overlap the others' reductions and epilogues.
#pragma once

#include <mutex>
#include <type_traits>

#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace mb {

constexpr int kCtaMaxThreads = 1024;
constexpr int kWideThreads = 512;  // CTA bound of the cluster kernels holding 32+ values per thread
constexpr int kWarpBlock = 256;
constexpr int kHdrBytes = 1024;   // reduction buffers, abort flags, mbarriers
constexpr int kMaxStages = 16;
constexpr int kMaxRowsInFlight = 8;  // resident CTAs per SM the planner aims for, at most
constexpr int kCappedRegs = 40;   // registers per thread of rows_cta_kernel_capped
// Local memory per thread (spilled registers) that the planners accept
// without preferring another launch: a few bytes (a value kept across the row
// loop, as in the two-slot bf16 LayerNorm kernel at 32 registers) cost nothing
// measurable; the forms they pass over spill hundreds.
constexpr size_t kSpillTolerance = 64;
// The same for the shifted-vector kernel, whose forms keep 16-20 bytes (the
// dropout chains' four-slot forms, measured no slower than the others) or
// spill 60 and more (eight slots of LayerNorm + residual, fp32 rows of 6147:
// 30% slower at three CTAs an SM than two CTAs of two slots without spills).
constexpr size_t kShiftSpillTolerance = 32;
// Bytes of row reads and writes per SM in flight that keep HBM busy; the
// planner aims for this many bytes' worth of resident rows, rounded to the
// nearest row count (sweeps on GB300, fp32: LayerNorm rows of 48 KB in + out
// fastest three to an SM, softmax rows of 32 KB four, causal score rows of
// 24 KB read + written five; bf16, whose rows carry twice the arithmetic per
// byte: LayerNorm rows of 48 KB four, 16 KB softmax rows eight).
constexpr int64_t kFlightBytesF32 = 128 * 1024;
constexpr int64_t kFlightBytesBf16 = 192 * 1024;
constexpr int kMaxCluster = 16;   // CTAs per row on the cluster path (above 8: opt-in size)
constexpr int kClusterRing = 1;   // staging ring depth on the cluster path (bf16)
constexpr int64_t kClusterStageMin = 64 * 1024;   // slices staged from this size (C::kStageLargeSlices)
constexpr int64_t kUnboundedRows = (int64_t)1 << 40;   // row count the cached plans assume

// Folds one slot's VEC values into the running first-pass partial (a sum, or a
// maximum with C::kMaxFirst); slots past the row end leave it unchanged.
template <class C, int VEC>
__device__ __forceinline__ float fold1(float acc, const float (&v)[VEC], bool valid) {
    if constexpr (C::kMaxFirst) {
        float m = v[0];
#pragma unroll
        for (int e = 1; e < VEC; ++e) m = fmaxf(m, v[e]);
        return valid ? fmaxf(acc, m) : acc;
    } else if constexpr (VEC == 1) {
        return acc + (valid ? v[0] : 0.0f);
    } else {
        float2 p = make_float2(v[0], v[1]);
#pragma unroll
        for (int e = 2; e < VEC; e += 2) p = add2(p, make_float2(v[e], v[e + 1]));
        return acc + (valid ? p.x + p.y : 0.0f);
    }
}

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
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows;
         row += nw) {
        const int64_t base = row * cols;
        // Every load of the row and of its per-column values is issued before
        // any is used: slots past the row end re-read the last vector (in
        // bounds) and are masked below.
        Frag<T, VEC> in[VPL][NIN];
        typename C::template PrePC<VEC> pre[VPL];
        typename C::template PostPC<VEC> post[VPL];
        const int ext = C::kPartialRows ? C::row_extent(a, row, cols) : cols;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int vc = min(lane + 32 * k, nvec - 1);
#pragma unroll
            for (int i = 0; i < NIN; ++i)
                in[k][i].load_stream_if(a.in[i] + base + vc * VEC, !C::kPartialRows || vc * VEC < ext);
            C::template load_pre<VEC>(a, vc * VEC, pre[k]);
            C::template load_post<VEC>(a, vc * VEC, post[k]);
        }
        typename C::template Early<VEC> ea[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k)
            C::template early<VEC>(a, base + min(lane + 32 * k, nvec - 1) * VEC, ea[k]);
        float v[VPL][VEC];
        float l1 = C::kMaxFirst ? -INFINITY : 0.0f;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            C::template pre<VEC>(in[k], pre[k], a, row, (lane + 32 * k) * VEC, v[k]);
            l1 = fold1<C, VEC>(l1, v[k], lane + 32 * k < nvec);
            if constexpr (C::kStorePre) {
                if (lane + 32 * k < nvec) C::template store_pre<VEC>(v[k], a, base + (lane + 32 * k) * VEC);
            }
        }
        const float mean = C::stat1(C::kMaxFirst ? warp_max(l1) : warp_sum(l1), cols, a);
        float rstd = 0.0f;
        if constexpr (C::kTwoPass) {
            float l2 = 0.0f;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const float part = C::template p2<VEC>(v[k], mean);
                l2 += lane + 32 * k < nvec ? part : 0.0f;
            }
            rstd = C::stat2(warp_sum(l2), cols, a);
        }
        if (lane == 0) C::store_stats(a, row, mean, rstd);
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int vi = lane + 32 * k;
            if (vi < nvec) {
                Frag<T, VEC> o;
                C::template post<VEC>(v[k], mean, rstd, post[k], a, base + vi * VEC, ea[k], o.f);
                o.store_stream(a.out + base + vi * VEC);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// one CTA per row, persistent; DIRECT or STAGED (bulk-async shared ring)
// ---------------------------------------------------------------------------
template <class C, int VPT, int VEC, bool STAGED>
__device__ __forceinline__ void rows_cta_body(const typename C::Args &a, int64_t rows, int cols,
                                              int nstage, unsigned *err) {
    using T = typename C::T;
    constexpr int NIN = C::kInputs;
    // The epilogue's per-column values are loaded with the row (before the
    // reduction barriers) only when that costs at most 8 registers: the
    // streaming shapes gain more from registers (CTAs per SM) than from the
    // earlier loads, which hit L1 anyway.
    constexpr bool kEarlyPost = VPT * VEC * C::kPostPC <= 8;
    using PrePC = typename C::template PrePC<VEC>;
    using PostPC = typename C::template PostPC<VEC>;
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
    pdl_wait();                 // the predecessor's writes are visible after this
    pdl_launch_dependents();
    __syncthreads();

    // Refill ring slot s with local row li (one elected thread).
    auto issue = [&](int s, int64_t li) {
        const int64_t row = first + li * G;
        const uint32_t bar = smem_addr(&bars[s]);
        // the row's first row_extent() elements, rounded up to 16 bytes
        // (rows hold a whole number of 16-byte vectors on this path)
        uint32_t bytes = ((uint32_t)C::row_extent(a, row, cols) * (uint32_t)sizeof(T) + 15u) & ~15u;
        if (bytes > row_bytes) bytes = row_bytes;
        mbar_arrive_expect_tx(bar, (uint32_t)NIN * bytes);
#pragma unroll
        for (int i = 0; i < NIN; ++i)
            bulk_g2s(smem_addr(ring + (size_t)s * stage_bytes + (size_t)i * row_bytes),
                     a.in[i] + row * cols, bytes, bar);
    };
    if constexpr (STAGED) {
        if (tid == 0) {
            const int64_t n0 = nlocal < nstage ? nlocal : nstage;
            for (int s = 0; s < (int)n0; ++s) issue(s, s);
        }
    }

    int rb = 0;
    int s = 0;              // ring slot of row li (li mod nstage)
    uint32_t parity = 0;    // barrier phase parity of row li ((li / nstage) & 1)
    int64_t li = 0;
    for (; li < nlocal; ++li) {
        const int64_t row = first + li * G;
        const int64_t base = row * cols;
        const T *stage = reinterpret_cast<const T *>(ring + (size_t)s * stage_bytes);

        // Per-column values first (they do not depend on the ring), then the
        // row: all loads before any use.  Slots past the row end re-read the
        // last vector and are masked.
        PrePC pre[VPT];
        PostPC post[kEarlyPost ? VPT : 1];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vc = min(tid + k * (int)blockDim.x, nvec - 1);
            C::template load_pre<VEC>(a, vc * VEC, pre[k]);
            if constexpr (kEarlyPost) C::template load_post<VEC>(a, vc * VEC, post[k]);
        }
        // values the epilogue needs that do not depend on the row's data,
        // drawn while the row is still in flight
        typename C::template Early<VEC> ea[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k)
            C::template early<VEC>(a, base + min(tid + k * (int)blockDim.x, nvec - 1) * VEC, ea[k]);
        if constexpr (STAGED) {
            if (!mbar_wait_bounded(smem_addr(&bars[s]), parity)) abort_flag[li & 1] = 1;
        }
        Frag<T, VEC> in[VPT][NIN];
        const int ext = C::kPartialRows && !STAGED ? C::row_extent(a, row, cols) : cols;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vc = min(tid + k * (int)blockDim.x, nvec - 1);
#pragma unroll
            for (int i = 0; i < NIN; ++i) {
                if constexpr (STAGED) in[k][i].load_shared(stage + (size_t)i * cols + vc * VEC);
                else in[k][i].load_stream_if(a.in[i] + base + vc * VEC,
                                             !C::kPartialRows || vc * VEC < ext);
            }
        }
        float v[VPT][VEC];
        float l1 = C::kMaxFirst ? -INFINITY : 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            C::template pre<VEC>(in[k], pre[k], a, row, (tid + k * (int)blockDim.x) * VEC, v[k]);
            l1 = fold1<C, VEC>(l1, v[k], tid + k * (int)blockDim.x < nvec);
            if constexpr (C::kStorePre) {
                const int vi = tid + k * (int)blockDim.x;
                if (vi < nvec) C::template store_pre<VEC>(v[k], a, base + vi * VEC);
            }
        }
        // Barrier inside: after it every thread has its row slice in registers.
        const float r1 = C::kMaxFirst ? block_max(l1, red + 32 * rb) : block_sum(l1, red + 32 * rb);
        rb ^= 1;
        if constexpr (STAGED) {
            if (abort_flag[li & 1]) break;
            if (tid == 0 && li + nstage < nlocal) issue(s, li + nstage);
        }
        const float mean = C::stat1(r1, cols, a);
        float rstd = 0.0f;
        if constexpr (C::kTwoPass) {
            float l2 = 0.0f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const float part = C::template p2<VEC>(v[k], mean);
                l2 += tid + k * (int)blockDim.x < nvec ? part : 0.0f;
            }
            rstd = C::stat2(block_sum(l2, red + 32 * rb), cols, a);
            rb ^= 1;
        }
        if (tid == 0) C::store_stats(a, row, mean, rstd);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vi = tid + k * blockDim.x;
            if (vi < nvec) {
                Frag<T, VEC> o;
                if constexpr (kEarlyPost) {
                    C::template post<VEC>(v[k], mean, rstd, post[k], a, base + vi * VEC, ea[k], o.f);
                } else {
                    PostPC pc;
                    C::template load_post<VEC>(a, vi * VEC, pc);
                    C::template post<VEC>(v[k], mean, rstd, pc, a, base + vi * VEC, ea[k], o.f);
                }
                o.store_stream(a.out + base + vi * VEC);
            }
        }
        if (++s == nstage) {
            s = 0;
            parity ^= 1u;
        }
    }
    if constexpr (STAGED) {
        // Only after a timed-out wait: record it, and wait (bounded) for this
        // CTA's copies still in flight before its shared memory goes away.
        if (li < nlocal && tid == 0) {
            atomicOr(err, kDevErrWaitTimeout);
            int ss = s;
            uint32_t pp = parity;
            for (int64_t lj = li; lj < nlocal && lj < li + nstage; ++lj) {
                (void)mbar_wait_bounded(smem_addr(&bars[ss]), pp);
                if (++ss == nstage) {
                    ss = 0;
                    pp ^= 1u;
                }
            }
        }
    }
}

template <class C, int VPT, int VEC, bool STAGED>
__global__ void __launch_bounds__(kCtaMaxThreads)
rows_cta_kernel(const typename C::Args a, int64_t rows, int cols, int nstage, unsigned *err) {
    rows_cta_body<C, VPT, VEC, STAGED>(a, rows, cols, nstage, err);
}

// The same engine bounded at kWideThreads threads, so a thread may hold up to
// 128 registers: the scalar (unaligned-row) forms with many slots per thread
// (C::kWideScalarSlots), which spill under the 64 registers of the
// 1024-thread bound.
template <class C, int VPT, int VEC, bool STAGED>
__global__ void __launch_bounds__(kWideThreads)
rows_cta_kernel_wide(const typename C::Args a, int64_t rows, int cols, int nstage, unsigned *err) {
    rows_cta_body<C, VPT, VEC, STAGED>(a, rows, cols, nstage, err);
}

// The same engine with the registers per thread capped (chains with
// C::kRegCap): more CTAs resident per SM for latency-bound chains.
template <class C, int VPT, int VEC, bool STAGED>
__global__ void __maxnreg__(kCappedRegs)
rows_cta_kernel_capped(const typename C::Args a, int64_t rows, int cols, int nstage, unsigned *err) {
    rows_cta_body<C, VPT, VEC, STAGED>(a, rows, cols, nstage, err);
}

// ---------------------------------------------------------------------------
// one CTA per row, rows off the 16-byte grid (shifted vectors)
// ---------------------------------------------------------------------------
// Rows whose length is not a whole number of vectors, or whose tensors do not
// start on a 16-byte boundary, when every row tensor (inputs, outputs) starts
// at the same offset m0 within 16 bytes: each row splits into a head of h <
// VEC elements up to its first 16-byte boundary, whole vectors from there,
// and a tail of fewer than VEC elements.  The vectors take the vector hooks
// with 16-byte row accesses; the head and tail elements take the scalar hooks,
// one element per thread.  Persistent over rows like rows_cta_kernel's direct
// path; the host guarantees cols >= 2 * VEC, so every row holds at least one
// whole vector.
// A vector slot's per-column values start at column h + k * VEC, off the
// 16-byte grid of the arrays.  Without CS they are loaded element by element;
// with CS the CTA copies every per-column array, from column h on, into
// shared memory (after the reduction header, each copy 16-byte aligned and
// `cstride` elements long), so a slot's values are 16-byte shared-memory
// loads.  The copy is made of 4-byte cp.async copies issued just before the
// row's loads, so it lands while they are in flight; each thread waits for
// its own copies before the first reduction, whose barrier publishes them
// (chains with per-column values before the reduction wait, and take a
// barrier, ahead of those loads).  h depends only on the row, and a grid of G
// CTAs keeps each CTA on one h when G * cols * sizeof(T) is a multiple of 16
// (the host rounds the grid so where the SM count allows); the copy is
// redone, behind a barrier, whenever a CTA's h changes.  The host plans CS
// for launches of several rows a CTA only (one row a CTA would copy as many
// values as it reads).
// STG (with CS, which copies nothing for chains without per-column arrays):
// the rows' whole vectors are streamed into a ring of nstage shared-memory
// stages after the copies, by bulk copies, as on rows_cta_kernel's staged
// path: a row's vector body starts on a 16-byte boundary and is a whole
// number of 16-byte words, so one bulk copy per input moves it, and a stage
// is refilled for the CTA's next row once the first reduction's barrier
// shows every thread holds the current one.  Head and tail elements stay
// plain loads, taken (with the values the epilogue draws early) before the
// stage wait, which their work hides.  Waits are bounded; a timeout ends the
// CTA's row loop after its copies in flight have landed and is reported in
// `err`.  The fourth argument then carries m0 | nstage << 8.
template <class C, int VPT, bool CS = false, bool STG = false>
__global__ void __launch_bounds__(kCtaMaxThreads)
rows_shift_kernel(const typename C::Args a, int64_t rows, int cols, int m0_arg, unsigned *err) {
    static_assert(!STG || CS, "the staged form is planned with the per-column copies");
    using T = typename C::T;
    constexpr int VEC = C::kVec;
    constexpr int NIN = C::kInputs;
    constexpr int ES = (int)sizeof(T);
    const int m0 = m0_arg & 15;
    const int nstage = STG ? m0_arg >> 8 : 0;
    // with CS the epilogue reads its values from shared memory, and only
    // chains with values before the reduction (kPreCols) wait for the copy
    // ahead of it; the others let the first reduction's barrier publish it
    constexpr bool kEarlyPost = !CS && VPT * VEC * C::kPostPC <= 8;
    using PrePC = typename C::template PrePC<VEC>;
    using PostPC = typename C::template PostPC<VEC>;
    using PrePC1 = typename C::template PrePC<1>;
    using PostPC1 = typename C::template PostPC<1>;
    constexpr bool kPreCols = !std::is_empty_v<PrePC>;
    extern __shared__ __align__(1024) unsigned char smem[];
    float *red = reinterpret_cast<float *>(smem);                  // [2][32]
    volatile int *abort_flag = reinterpret_cast<int *>(smem + 256); // STG: [2]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 512);     // STG: [kMaxStages]
    T *cs = reinterpret_cast<T *>(smem + kHdrBytes);   // CS: [kColArrays][cstride]
    const int cstride = (cols + 15) & ~15;
    // STG: the ring, [nstage][NIN][cstride] after the per-column copies
    unsigned char *ring = smem + kHdrBytes + (size_t)C::kColArrays * cstride * ES;
    const uint32_t stage_bytes = (uint32_t)NIN * (uint32_t)cstride * (uint32_t)ES;
    const int tid = threadIdx.x;
    const int T_ = (int)blockDim.x;
    const int64_t G = gridDim.x;
    const int64_t first = blockIdx.x;
    const int64_t nlocal = STG && first < rows ? (rows - first + G - 1) / G : 0;   // STG
    if constexpr (STG) {
        if (tid == 0) {
            abort_flag[0] = 0;
            abort_flag[1] = 0;
            for (int q = 0; q < nstage; ++q) mbar_init(smem_addr(&bars[q]), 1);
            fence_mbar_init();
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    // STG: refill stage q with local row li's whole vectors (one elected thread)
    auto issue = [&](int q, int64_t li) {
        const int64_t row = first + li * G;
        const int64_t base = row * cols;
        const int off = (int)(((uint64_t)m0 + (uint64_t)base * (uint64_t)ES) & 15u);
        const int h = ((16 - off) & 15) / ES;
        const uint32_t bytes = (uint32_t)((cols - h) / VEC * VEC) * (uint32_t)ES;
        const uint32_t bar = smem_addr(&bars[q]);
        mbar_arrive_expect_tx(bar, (uint32_t)NIN * bytes);
#pragma unroll
        for (int i = 0; i < NIN; ++i)
            bulk_g2s(smem_addr(ring + (size_t)q * stage_bytes + (size_t)i * cstride * ES),
                     a.in[i] + base + h, bytes, bar);
    };
    if constexpr (STG) {
        __syncthreads();        // the barriers are initialised
        if (tid == 0) {
            const int64_t n0 = nlocal < nstage ? nlocal : nstage;
            for (int q = 0; q < (int)n0; ++q) issue(q, q);
        }
    }
    int rb = 0;
    int hs = -1;                                               // CS: h of the copy held
    int sq = 0;                 // STG: ring stage of local row li
    uint32_t parity = 0;        // STG: its phase parity
    int64_t li = 0;             // STG: the CTA's rows done
    for (int64_t row = first; row < rows; row += G) {
        const int64_t base = row * cols;
        // the row's first element sits `off` bytes past a 16-byte boundary
        const int off = (int)(((uint64_t)m0 + (uint64_t)base * (uint64_t)ES) & 15u);
        const int h = ((16 - off) & 15) / ES;                  // head elements
        const int nb = (cols - h) / VEC;                       // whole vectors (>= 1)
        const auto vld = [&] {
            if constexpr (CS) return ColsShared<T>{cs, cstride, h};
            else return ColsGlobal<false>{};
        }();
        const int ne = cols - nb * VEC;                        // head + tail elements
        const int ext = C::kPartialRows ? C::row_extent(a, row, cols) : cols;
        const bool has_e = tid < ne;
        const int col_e = tid < h ? tid : h + nb * VEC + (tid - h);
        const int64_t vbase = base + h;                        // first whole vector

        // CS: a CTA meeting a new h starts its per-column copy (asynchronous
        // 4-byte copies, no registers held while they fly; bf16 arrays whose
        // column h is not 4-byte aligned are copied element by element)
        const bool restage = CS && h != hs;                    // uniform across the CTA
        if constexpr (CS) {
            if (restage) {
                if (hs >= 0) __syncthreads();   // every read of the old copy is done
                const int n = cols - h;
#pragma unroll
                for (int i = 0; i < C::kColArrays; ++i) {
                    const T *src = C::col_array(a, i) + h;
                    T *dst = cs + i * cstride;
                    if (ES == 4 || (reinterpret_cast<uintptr_t>(src) & 3u) == 0) {
                        constexpr int PER = 4 / ES;             // elements per copy
                        for (int m = tid; m < n / PER; m += T_)
                            cp_async4(smem_addr(dst + m * PER), src + m * PER);
                        if (PER == 2 && (n & 1) && tid == 0) dst[n - 1] = src[n - 1];
                    } else {
                        for (int j = tid; j < n; j += T_) dst[j] = src[j];
                    }
                }
            }
        }
        // every load before any use; vector slots past the row's last vector
        // re-read it (in bounds) and are masked below
        PrePC pre[VPT];
        PostPC post[kEarlyPost ? VPT : 1];
        Frag<T, VEC> in[VPT][NIN];
        PrePC1 pre_e;
        PostPC1 post_e;
        Frag<T, 1> in_e[NIN];
        typename C::template Early<VEC> ea[VPT];
        typename C::template Early<1> ea_e;
        if constexpr (STG) {
            // head and tail elements, and the values the epilogue needs that
            // do not depend on the row's data, before the ring wait (their
            // work hides it); the unstaged form takes them after its loads
            if (has_e) {
                C::template load_pre<1>(a, col_e, pre_e);
                C::template load_post<1>(a, col_e, post_e);
#pragma unroll
                for (int i = 0; i < NIN; ++i) in_e[i].load_stream(a.in[i] + base + col_e);
            } else {
#pragma unroll
                for (int i = 0; i < NIN; ++i) in_e[i].f[0] = 0.0f;
            }
#pragma unroll
            for (int k = 0; k < VPT; ++k)
                C::template early<VEC, true>(a, vbase + (int64_t)min(tid + k * T_, nb - 1) * VEC,
                                             ea[k]);
            C::template early<1>(a, base + (has_e ? col_e : 0), ea_e);
        }
        const T *stage = nullptr;
        if constexpr (STG) {
            if (!mbar_wait_bounded(smem_addr(&bars[sq]), parity)) abort_flag[li & 1] = 1;
            stage = reinterpret_cast<const T *>(ring + (size_t)sq * stage_bytes);
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vc = min(tid + k * T_, nb - 1);
            if constexpr (!CS) {
                C::template load_pre<VEC>(a, h + vc * VEC, pre[k], vld);
                if constexpr (kEarlyPost) C::template load_post<VEC>(a, h + vc * VEC, post[k], vld);
            }
#pragma unroll
            for (int i = 0; i < NIN; ++i) {
                if constexpr (STG) in[k][i].load_shared(stage + (size_t)i * cstride + vc * VEC);
                else in[k][i].load_stream_if(a.in[i] + vbase + (int64_t)vc * VEC,
                                             !C::kPartialRows || h + vc * VEC < ext);
            }
        }
        if constexpr (CS && kPreCols) {
            // the copies land while the row's loads are in flight
            if (restage) {
                cp_async_wait_all();
                __syncthreads();
            }
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int vc = min(tid + k * T_, nb - 1);
                C::template load_pre<VEC>(a, h + vc * VEC, pre[k], vld);
            }
        }
        if constexpr (!STG) {
            if (has_e) {
                C::template load_pre<1>(a, col_e, pre_e);
                C::template load_post<1>(a, col_e, post_e);
#pragma unroll
                for (int i = 0; i < NIN; ++i)
                    in_e[i].load_stream_if(a.in[i] + base + col_e,
                                           !C::kPartialRows || col_e < ext);
            } else {
#pragma unroll
                for (int i = 0; i < NIN; ++i) in_e[i].f[0] = 0.0f;
            }
#pragma unroll
            for (int k = 0; k < VPT; ++k)
                C::template early<VEC, true>(a, vbase + (int64_t)min(tid + k * T_, nb - 1) * VEC,
                                             ea[k]);
            C::template early<1>(a, base + (has_e ? col_e : 0), ea_e);
        }

        float v[VPT][VEC];
        float ve[1];
        float l1 = C::kMaxFirst ? -INFINITY : 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vi = tid + k * T_;
            C::template pre<VEC>(in[k], pre[k], a, row, h + vi * VEC, v[k]);
            l1 = fold1<C, VEC>(l1, v[k], vi < nb);
            if constexpr (C::kStorePre) {
                if (vi < nb) C::template store_pre<VEC>(v[k], a, vbase + (int64_t)vi * VEC);
            }
        }
        C::template pre<1>(in_e, pre_e, a, row, has_e ? col_e : 0, ve);
        l1 = fold1<C, 1>(l1, ve, has_e);
        if constexpr (C::kStorePre) {
            if (has_e) C::template store_pre<1>(ve, a, base + col_e);
        }
        if constexpr (CS) {
            // this thread's copies are done; the reduction's barrier makes
            // every thread's visible before the epilogue reads them
            if (restage) {
                if constexpr (!kPreCols) cp_async_wait_all();
                hs = h;
            }
        }
        const float r1 = C::kMaxFirst ? block_max(l1, red + 32 * rb) : block_sum(l1, red + 32 * rb);
        rb ^= 1;
        if constexpr (STG) {
            // after the barrier every thread holds its part of the row
            if (abort_flag[li & 1]) break;
            if (tid == 0 && li + nstage < nlocal) issue(sq, li + nstage);
        }
        const float mean = C::stat1(r1, cols, a);
        float rstd = 0.0f;
        if constexpr (C::kTwoPass) {
            float l2 = 0.0f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const float part = C::template p2<VEC>(v[k], mean);
                l2 += tid + k * T_ < nb ? part : 0.0f;
            }
            const float part_e = C::template p2<1>(ve, mean);
            l2 += has_e ? part_e : 0.0f;
            rstd = C::stat2(block_sum(l2, red + 32 * rb), cols, a);
            rb ^= 1;
        }
        if (tid == 0) C::store_stats(a, row, mean, rstd);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vi = tid + k * T_;
            if (vi < nb) {
                Frag<T, VEC> o;
                if constexpr (kEarlyPost) {
                    C::template post<VEC>(v[k], mean, rstd, post[k], a, vbase + (int64_t)vi * VEC,
                                          ea[k], o.f);
                } else {
                    PostPC pc;
                    C::template load_post<VEC>(a, h + vi * VEC, pc, vld);
                    C::template post<VEC>(v[k], mean, rstd, pc, a, vbase + (int64_t)vi * VEC,
                                          ea[k], o.f);
                }
                o.store_stream(a.out + vbase + (int64_t)vi * VEC);
            }
        }
        if (has_e) {
            Frag<T, 1> o;
            C::template post<1>(ve, mean, rstd, post_e, a, base + col_e, ea_e, o.f);
            o.store_stream(a.out + base + col_e);
        }
        if constexpr (STG) {
            if (++sq == nstage) {
                sq = 0;
                parity ^= 1u;
            }
            ++li;
        }
    }
    if constexpr (STG) {
        // Only after a timed-out wait: record it, and wait (bounded) for this
        // CTA's copies still in flight before its shared memory goes away.
        if (li < nlocal && tid == 0) {
            atomicOr(err, kDevErrWaitTimeout);
            int qq = sq;
            uint32_t pp = parity;
            for (int64_t lj = li; lj < nlocal && lj < li + nstage; ++lj) {
                (void)mbar_wait_bounded(smem_addr(&bars[qq]), pp);
                if (++qq == nstage) {
                    qq = 0;
                    pp ^= 1u;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// one thread-block cluster per row (rows longer than one CTA can hold)
// ---------------------------------------------------------------------------

// Sum (or maximum) of one value per CTA over the cluster.  Thread 0 pushes
// this CTA's partial into slot `rank` of every CTA's exchange buffer `xch`
// (kMaxCluster floats) with st.async, which completes 4 transaction bytes on
// that CTA's mbarrier `bar`; every CTA arms its own mbarrier for cs pushes,
// waits on it (bounded; a timeout sets *abort) and folds the slots in rank
// order, so all CTAs get the bitwise-same value.  No cluster barrier: its
// release half would first wait for every load and store this thread has in
// flight (the next row's prefetch, this row's stores), serialising them with
// the exchange.  Two buffers alternate between reductions; a CTA pushes into
// buffer b again only after every CTA has pushed the reduction in between,
// which each does after reading b.
template <bool MAX>
__device__ __forceinline__ float cluster_reduce(float v, float *xch, uint64_t *bar,
                                                uint32_t &parity, unsigned cs, unsigned rank,
                                                volatile int *abort) {
    const uint32_t bar_a = smem_addr(bar);
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx_relaxed(bar_a, cs * 4u);
        const uint32_t slot = smem_addr(xch + rank);
        for (unsigned j = 0; j < cs; ++j) st_async_f32(map_cluster(slot, j), v, map_cluster(bar_a, j));
    }
    if (!mbar_wait_bounded(bar_a, parity)) *abort = 1;
    parity ^= 1u;
    float r = MAX ? -INFINITY : 0.0f;
    for (unsigned j = 0; j < cs; ++j) {
        const float p = xch[j];
        r = MAX ? fmaxf(r, p) : r + p;
    }
    return r;
}

// The cluster of CS CTAs owns rows c, c + nclusters, ...; CTA `rank` holds the
// columns [rank * slice, (rank + 1) * slice) of each of them in registers.
//   STAGED  one elected thread streams the CTA's slice of each row (every
//           input) into a ring of `nstage` shared-memory stages with bulk async
//           copies, as the one-CTA staged engine does; a stage is refilled as
//           soon as the first reduction barrier shows every thread holds its
//           row in registers.
//   DIRECT  vector loads, the next row's issued into registers as soon as the
//           current row has left them (unaligned rows, rows in host memory).
// The two statistics combine CTA partials through distributed shared memory
// (cluster_reduce).  Every wait is bounded; a timeout ends the CTA's row loop
// (after its copies in flight have landed) and is reported in `err`.
// MAXT bounds the CTA size: launches of 32 or more values per thread on at
// most kWideThreads threads take the kWideThreads form, whose threads may hold
// up to 128 registers (the slice, the next row's prefetch and the per-column
// values), where under the 64 of the 1024-thread form they spill.
// SH: rows off the 16-byte grid whose tensors share the offset m0 within 16
// bytes (the sixth argument carries m0 << 8 above the ring depth), as the
// shifted one-CTA kernel reads them: a row's head of h < VEC elements, its
// nb = (cols - h) / VEC whole vectors, of which CTA `rank` holds those from
// vector rank * slice / VEC on (as many as remain, up to slice / VEC; the
// host sizes slice for the most any row has), and its tail; the head and tail
// elements go to rank 0, one a thread.  The per-column values of a slot start
// off the arrays' 16-byte grid and are loaded element by element.
template <class C, int VPT, int VEC, bool STAGED, int MAXT, bool SH = false>
__global__ void __launch_bounds__(MAXT, 1)
rows_cluster_kernel(const typename C::Args a, int64_t rows, int cols, int slice, unsigned *err,
                    int nstage_arg) {
    static_assert(!SH || !C::kPartialRows, "shifted cluster rows are read whole");
    namespace cg = cooperative_groups;
    using T = typename C::T;
    constexpr int NIN = C::kInputs;
    constexpr int ES = (int)sizeof(T);
    const int nstage = SH ? nstage_arg & 255 : nstage_arg;
    const int m0 = SH ? (nstage_arg >> 8) & 15 : 0;
    using PrePC1 = typename C::template PrePC<1>;
    using PostPC1 = typename C::template PostPC<1>;
    constexpr bool kEarlyPost = VPT * VEC * C::kPostPC <= 8;
    using PrePC = typename C::template PrePC<VEC>;
    using PostPC = typename C::template PostPC<VEC>;
    extern __shared__ __align__(1024) unsigned char ring[];   // STAGED: [nstage][NIN][slice]
    __shared__ float red[2][32];
    __shared__ float xch[2][kMaxCluster];
    __shared__ __align__(8) uint64_t xbar[2];
    __shared__ __align__(8) uint64_t sbar[kMaxStages];
    __shared__ int stage_abort[2];    // a stage wait timed out (by row parity)
    __shared__ int xch_abort[2];      // an exchange wait timed out (by row parity)
    cg::cluster_group cl = cg::this_cluster();
    const int tid = threadIdx.x;
    const int rank = (int)cl.block_rank();
    const unsigned cs = cl.num_blocks();
    const int64_t nclusters = gridDim.x / cs;
    const int64_t cid = blockIdx.x / cs;
    const int lo = rank * slice;                               // first column of this CTA
    const int hi = lo + slice < cols ? lo + slice : cols;
    const int nvec = hi > lo ? (hi - lo) / VEC : 0;            // vectors this CTA holds
    const int64_t nlocal = cid < rows ? (rows - cid + nclusters - 1) / nclusters : 0;
    const uint32_t pitch = (uint32_t)slice * (uint32_t)sizeof(T);           // per input, in a stage
    const uint32_t my_bytes = (uint32_t)(nvec * VEC) * (uint32_t)sizeof(T);
    const uint32_t stage_bytes = (uint32_t)NIN * pitch;
    // SH: a row's head, and the whole vectors of it this CTA holds
    auto head_of = [&](int64_t row) -> int {
        if constexpr (SH) {
            const int off =
                (int)(((uint64_t)m0 + (uint64_t)row * (uint64_t)cols * (uint64_t)ES) & 15u);
            return ((16 - off) & 15) / ES;
        } else {
            return 0;
        }
    };
    auto nv_of = [&](int h) -> int {
        if constexpr (SH) {
            const int n = (cols - h) / VEC - lo / VEC;
            return n < 0 ? 0 : (n < slice / VEC ? n : slice / VEC);
        } else {
            return nvec;
        }
    };
    if (tid == 0) {
        mbar_init(smem_addr(&xbar[0]), 1);
        mbar_init(smem_addr(&xbar[1]), 1);
        if constexpr (STAGED) {
            for (int q = 0; q < nstage; ++q) mbar_init(smem_addr(&sbar[q]), 1);
        }
        stage_abort[0] = stage_abort[1] = 0;
        xch_abort[0] = xch_abort[1] = 0;
        fence_mbar_init();
    }
    cl.sync();      // every CTA's barriers are initialised before any push
    pdl_wait();
    pdl_launch_dependents();

    // STAGED: refill stage q with local row li (one elected thread).
    auto issue = [&](int q, int64_t li) {
        const int64_t row = cid + li * nclusters;
        const uint32_t bar = smem_addr(&sbar[q]);
        const int h = head_of(row);
        uint32_t bytes;
        if constexpr (SH) {
            // this rank's whole vectors of the row
            bytes = (uint32_t)(nv_of(h) * VEC) * (uint32_t)sizeof(T);
        } else {
            // this rank's part of the row's first row_extent() elements,
            // rounded up to whole vectors (16 or 32 bytes) within the slice
            const int ext = C::row_extent(a, row, cols) - lo;
            bytes = ext <= 0 ? 0u
                  : ((uint32_t)((ext + VEC - 1) / VEC) * VEC) * (uint32_t)sizeof(T);
            if (bytes > my_bytes) bytes = my_bytes;
        }
        mbar_arrive_expect_tx(bar, (uint32_t)NIN * bytes);
        if (bytes == 0) return;
#pragma unroll
        for (int i = 0; i < NIN; ++i)
            bulk_g2s(smem_addr(ring + (size_t)q * stage_bytes + (size_t)i * pitch),
                     a.in[i] + row * cols + h + lo, bytes, bar);
    };
    if constexpr (STAGED) {
        if (tid == 0) {
            const int64_t n0 = nlocal < nstage ? nlocal : nstage;
            for (int q = 0; q < (int)n0; ++q) issue(q, q);
        }
    }

    // Per-column values of the slots (and, DIRECT, the row's slice) for row
    // r; the planner leaves no rank empty, and indices stay in bounds
    // regardless.
    PrePC pre[VPT];
    PostPC post[kEarlyPost ? VPT : 1];
    Frag<T, VEC> in[VPT][NIN];
    // (SH: the row's head h and this CTA's vectors nv of it)
    auto load_cols = [&](int h, int nv) {
        if (nv == 0) return;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vc = min(tid + k * (int)blockDim.x, nv - 1);
            C::template load_pre<VEC>(a, h + lo + vc * VEC, pre[k], ColsGlobal<!SH>{});
            if constexpr (kEarlyPost)
                C::template load_post<VEC>(a, h + lo + vc * VEC, post[k], ColsGlobal<!SH>{});
        }
    };
    auto load_row = [&](int64_t r) {
        const int h = head_of(r);
        const int nv = nv_of(h);
        if (nv == 0) return;
        load_cols(h, nv);
        const int ext = C::kPartialRows ? C::row_extent(a, r, cols) : cols;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vc = min(tid + k * (int)blockDim.x, nv - 1);
#pragma unroll
            for (int i = 0; i < NIN; ++i)
                in[k][i].load_stream_if(a.in[i] + r * cols + h + lo + vc * VEC,
                                        !C::kPartialRows || lo + vc * VEC < ext);
        }
    };
    // SH: a row's head and tail elements, one a thread on rank 0.  Loaded at
    // the top of the row's iteration, where the staged path's wait or the
    // chain's first pass hides them; the direct path of a chain whose first
    // pass is a bare maximum (the softmax) loads them with the previous row
    // in flight instead (softmax fp32, 50257 columns: 82.0 us against 126.9;
    // the others ran 6-12% slower that way, the held values pushing the
    // 1024-thread forms into spills).
    constexpr bool kEdgesAhead = SH && !STAGED && C::kMaxFirst;
    Frag<T, 1> in_e[NIN];
    auto load_edges = [&](int64_t r) {
        if constexpr (SH) {
            const int h = head_of(r);
            const int nb = (cols - h) / VEC;
            const int col_e = tid < h ? tid : h + nb * VEC + (tid - h);
            if (rank == 0 && tid < cols - nb * VEC) {
#pragma unroll
                for (int i = 0; i < NIN; ++i) in_e[i].load_stream(a.in[i] + r * cols + col_e);
            } else {
#pragma unroll
                for (int i = 0; i < NIN; ++i) in_e[i].f[0] = 0.0f;
            }
        }
    };
    if constexpr (kEdgesAhead) {
        if (nlocal > 0) load_edges(cid);
    }
    if constexpr (!STAGED) {
        if (nlocal > 0) load_row(cid);
    }

    int rb = 0, xb = 0;
    uint32_t xpar[2] = {0u, 0u};
    int q = 0;                  // ring stage of local row li
    uint32_t parity = 0;        // its phase parity
    int64_t li = 0;
    for (; li < nlocal; ++li) {
        const int64_t row = cid + li * nclusters;
        const int h = head_of(row);                            // SH; else 0
        const int nvr = nv_of(h);                              // SH: this row's; else nvec
        const int64_t base = row * cols + h + lo;
        typename C::template Early<VEC> ea[VPT];
        if (nvr > 0) {
#pragma unroll
            for (int k = 0; k < VPT; ++k)
                C::template early<VEC, SH>(a, base + min(tid + k * (int)blockDim.x, nvr - 1) * VEC,
                                           ea[k]);
        }
        // SH: the row's head and tail elements, one a thread on rank 0
        const int nb = SH ? (cols - h) / VEC : 0;
        const bool has_e = SH && rank == 0 && tid < cols - nb * VEC;
        const int col_e = tid < h ? tid : h + nb * VEC + (tid - h);
        PrePC1 pre_e;
        PostPC1 post_e;
        typename C::template Early<1> ea_e;
        if constexpr (SH) {
            if constexpr (!kEdgesAhead) load_edges(row);
            if (has_e) {
                C::template load_pre<1>(a, col_e, pre_e);
                C::template load_post<1>(a, col_e, post_e);
            }
            C::template early<1>(a, row * cols + (has_e ? col_e : 0), ea_e);
        }
        if constexpr (STAGED) {
            load_cols(h, nvr);
            if (!mbar_wait_bounded(smem_addr(&sbar[q]), parity)) stage_abort[li & 1] = 1;
            const T *stage = reinterpret_cast<const T *>(ring + (size_t)q * stage_bytes);
            if (nvr > 0) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int vc = min(tid + k * (int)blockDim.x, nvr - 1);
#pragma unroll
                    for (int i = 0; i < NIN; ++i)
                        in[k][i].load_shared(stage + (size_t)i * slice + vc * VEC);
                }
            }
        }
        float v[VPT][VEC];
        float ve[1];
        float l1 = C::kMaxFirst ? -INFINITY : 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vi = tid + k * (int)blockDim.x;
            C::template pre<VEC>(in[k], pre[k], a, row, h + lo + vi * VEC, v[k]);
            l1 = fold1<C, VEC>(l1, v[k], vi < nvr);
            if constexpr (C::kStorePre) {
                if (vi < nvr) C::template store_pre<VEC>(v[k], a, base + vi * VEC);
            }
        }
        if constexpr (SH) {
            C::template pre<1>(in_e, pre_e, a, row, has_e ? col_e : 0, ve);
            l1 = fold1<C, 1>(l1, ve, has_e);
            if constexpr (C::kStorePre) {
                if (has_e) C::template store_pre<1>(ve, a, row * cols + col_e);
            }
            if constexpr (kEdgesAhead) {
                if (li + 1 < nlocal) load_edges(row + nclusters);
            }
        }
        // DIRECT: the input registers are free now, so the next row's loads
        // stay in flight through this row's reductions and epilogue.
        if constexpr (!STAGED) {
            if (li + 1 < nlocal) load_row(row + nclusters);
        }
        const float c1 = C::kMaxFirst ? block_max(l1, red[rb]) : block_sum(l1, red[rb]);
        rb ^= 1;
        // Timeouts: this row's stage wait, or an exchange of the previous row
        // (flags alternate by row, so every thread reads the same values here).
        if (stage_abort[li & 1] | xch_abort[(li + 1) & 1]) break;
        if constexpr (STAGED) {
            if (tid == 0 && li + nstage < nlocal) issue(q, li + nstage);
        }
        volatile int *ab = &xch_abort[li & 1];
        const float r1 = cluster_reduce<C::kMaxFirst>(c1, xch[xb], &xbar[xb], xpar[xb], cs, rank, ab);
        xb ^= 1;
        const float mean = C::stat1(r1, cols, a);
        float rstd = 0.0f;
        if constexpr (C::kTwoPass) {
            float l2 = 0.0f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const float part = C::template p2<VEC>(v[k], mean);
                l2 += tid + k * (int)blockDim.x < nvr ? part : 0.0f;
            }
            if constexpr (SH) {
                const float part_e = C::template p2<1>(ve, mean);
                l2 += has_e ? part_e : 0.0f;
            }
            const float c2 = block_sum(l2, red[rb]);
            rb ^= 1;
            rstd = C::stat2(cluster_reduce<false>(c2, xch[xb], &xbar[xb], xpar[xb], cs, rank, ab),
                            cols, a);
            xb ^= 1;
        }
        if (rank == 0 && tid == 0) C::store_stats(a, row, mean, rstd);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int vi = tid + k * blockDim.x;
            if (vi < nvr) {
                Frag<T, VEC> o;
                if constexpr (kEarlyPost) {
                    C::template post<VEC>(v[k], mean, rstd, post[k], a, base + vi * VEC, ea[k], o.f);
                } else {
                    PostPC pc;
                    C::template load_post<VEC>(a, h + lo + vi * VEC, pc, ColsGlobal<!SH>{});
                    C::template post<VEC>(v[k], mean, rstd, pc, a, base + vi * VEC, ea[k], o.f);
                }
                o.store_stream(a.out + base + vi * VEC);
            }
        }
        if constexpr (SH) {
            if (has_e) {
                Frag<T, 1> o;
                C::template post<1>(ve, mean, rstd, post_e, a, row * cols + col_e, ea_e, o.f);
                o.store_stream(a.out + row * cols + col_e);
            }
        }
        if constexpr (STAGED) {
            if (++q == nstage) {
                q = 0;
                parity ^= 1u;
            }
        }
    }
    if (tid == 0) {
        if (li < nlocal || (xch_abort[0] | xch_abort[1])) atomicOr(err, kDevErrWaitTimeout);
        if constexpr (STAGED) {
            // Only after a timeout: wait (bounded) for this CTA's copies still
            // in flight before its shared memory goes away.
            int qq = q;
            uint32_t pp = parity;
            for (int64_t lj = li; lj < nlocal && lj < li + nstage; ++lj) {
                (void)mbar_wait_bounded(smem_addr(&sbar[qq]), pp);
                if (++qq == nstage) {
                    qq = 0;
                    pp ^= 1u;
                }
            }
        }
    }
    cl.sync();     // no CTA leaves while another may still push into its slots
}

// Rows longer than a CTA, the CTA's slice held in shared memory rather than
// registers (bf16 rows of chains with C::kStageLargeSlices, slices of
// kClusterStageMin bytes or more): one elected thread streams the slice of
// each row into a ring of nstage stages with bulk async copies; every pass
// (the first statistic, the second, the epilogue) reads it back from the
// stage, so a thread holds one vector at a time and a CTA keeps 1024 threads
// at about 40 registers.  The second pass's in-place transform (p2) is
// applied again in the epilogue, so each value reaches `post` exactly as on
// the register path.  A stage is refilled once the epilogue of its row has
// read it.  Waits and exchanges are bounded as in rows_cluster_kernel.
template <class C, int VEC>
__global__ void __launch_bounds__(kCtaMaxThreads, 1)
rows_cluster_smem_kernel(const typename C::Args a, int64_t rows, int cols, int slice,
                         unsigned *err, int nstage) {
    namespace cg = cooperative_groups;
    using T = typename C::T;
    constexpr int NIN = C::kInputs;
    using PrePC = typename C::template PrePC<VEC>;
    using PostPC = typename C::template PostPC<VEC>;
    extern __shared__ __align__(1024) unsigned char ring[];   // [nstage][NIN][slice]
    __shared__ float red[2][32];
    __shared__ float xch[2][kMaxCluster];
    __shared__ __align__(8) uint64_t xbar[2];
    __shared__ __align__(8) uint64_t sbar[kMaxStages];
    __shared__ int stage_abort[2];
    __shared__ int xch_abort[2];
    cg::cluster_group cl = cg::this_cluster();
    const int tid = threadIdx.x;
    const int rank = (int)cl.block_rank();
    const unsigned cs = cl.num_blocks();
    const int64_t nclusters = gridDim.x / cs;
    const int64_t cid = blockIdx.x / cs;
    const int lo = rank * slice;
    const int hi = lo + slice < cols ? lo + slice : cols;
    const int nvec = hi > lo ? (hi - lo) / VEC : 0;
    const int64_t nlocal = cid < rows ? (rows - cid + nclusters - 1) / nclusters : 0;
    const uint32_t pitch = (uint32_t)slice * (uint32_t)sizeof(T);
    const uint32_t my_bytes = (uint32_t)(nvec * VEC) * (uint32_t)sizeof(T);
    const uint32_t stage_bytes = (uint32_t)NIN * pitch;
    if (tid == 0) {
        mbar_init(smem_addr(&xbar[0]), 1);
        mbar_init(smem_addr(&xbar[1]), 1);
        for (int q = 0; q < nstage; ++q) mbar_init(smem_addr(&sbar[q]), 1);
        stage_abort[0] = stage_abort[1] = 0;
        xch_abort[0] = xch_abort[1] = 0;
        fence_mbar_init();
    }
    cl.sync();
    pdl_wait();
    pdl_launch_dependents();
    auto issue = [&](int q, int64_t li) {
        const int64_t row = cid + li * nclusters;
        const uint32_t bar = smem_addr(&sbar[q]);
        const int ext = C::row_extent(a, row, cols) - lo;
        uint32_t bytes = ext <= 0 ? 0u
                       : ((uint32_t)((ext + VEC - 1) / VEC) * VEC) * (uint32_t)sizeof(T);
        if (bytes > my_bytes) bytes = my_bytes;
        mbar_arrive_expect_tx(bar, (uint32_t)NIN * bytes);
        if (bytes == 0) return;
#pragma unroll
        for (int i = 0; i < NIN; ++i)
            bulk_g2s(smem_addr(ring + (size_t)q * stage_bytes + (size_t)i * pitch),
                     a.in[i] + row * cols + lo, bytes, bar);
    };
    if (tid == 0) {
        const int64_t n0 = nlocal < nstage ? nlocal : nstage;
        for (int q = 0; q < (int)n0; ++q) issue(q, q);
    }
    int rb = 0, xb = 0;
    uint32_t xpar[2] = {0u, 0u};
    int q = 0;
    uint32_t parity = 0;
    int64_t li = 0;
    const int nthr = (int)blockDim.x;
    for (; li < nlocal; ++li) {
        const int64_t row = cid + li * nclusters;
        const int64_t base = row * cols + lo;
        if (!mbar_wait_bounded(smem_addr(&sbar[q]), parity)) stage_abort[li & 1] = 1;
        const T *stage = reinterpret_cast<const T *>(ring + (size_t)q * stage_bytes);
        // v of vector vi of the slice (the prologue applied)
        auto value = [&](int vi, float (&v)[VEC]) {
            Frag<T, VEC> in[NIN];
#pragma unroll
            for (int i = 0; i < NIN; ++i) in[i].load_shared(stage + (size_t)i * slice + vi * VEC);
            PrePC pc;
            C::template load_pre<VEC>(a, lo + vi * VEC, pc);
            C::template pre<VEC>(in, pc, a, row, lo + vi * VEC, v);
        };
        float l1 = C::kMaxFirst ? -INFINITY : 0.0f;
        for (int vi = tid; vi < nvec; vi += nthr) {
            float v[VEC];
            value(vi, v);
            l1 = fold1<C, VEC>(l1, v, true);
            if constexpr (C::kStorePre) C::template store_pre<VEC>(v, a, base + vi * VEC);
        }
        const float c1 = C::kMaxFirst ? block_max(l1, red[rb]) : block_sum(l1, red[rb]);
        rb ^= 1;
        if (stage_abort[li & 1] | xch_abort[(li + 1) & 1]) break;
        volatile int *ab = &xch_abort[li & 1];
        const float r1 = cluster_reduce<C::kMaxFirst>(c1, xch[xb], &xbar[xb], xpar[xb], cs, rank, ab);
        xb ^= 1;
        const float mean = C::stat1(r1, cols, a);
        float rstd = 0.0f;
        if constexpr (C::kTwoPass) {
            float l2 = 0.0f;
            for (int vi = tid; vi < nvec; vi += nthr) {
                float v[VEC];
                value(vi, v);
                l2 += C::template p2<VEC>(v, mean);
            }
            const float c2 = block_sum(l2, red[rb]);
            rb ^= 1;
            rstd = C::stat2(cluster_reduce<false>(c2, xch[xb], &xbar[xb], xpar[xb], cs, rank, ab),
                            cols, a);
            xb ^= 1;
        }
        if (rank == 0 && tid == 0) C::store_stats(a, row, mean, rstd);
        for (int vi = tid; vi < nvec; vi += nthr) {
            float v[VEC];
            value(vi, v);
            if constexpr (C::kTwoPass) (void)C::template p2<VEC>(v, mean);
            typename C::template Early<VEC> ea;
            C::template early<VEC>(a, base + vi * VEC, ea);
            PostPC pc;
            C::template load_post<VEC>(a, lo + vi * VEC, pc);
            Frag<T, VEC> o;
            C::template post<VEC>(v, mean, rstd, pc, a, base + vi * VEC, ea, o.f);
            o.store_stream(a.out + base + vi * VEC);
        }
        // every thread has read the stage: refill it with row li + nstage
        __syncthreads();
        if (tid == 0 && li + nstage < nlocal) issue(q, li + nstage);
        if (++q == nstage) {
            q = 0;
            parity ^= 1u;
        }
    }
    if (tid == 0) {
        if (li < nlocal || (xch_abort[0] | xch_abort[1])) atomicOr(err, kDevErrWaitTimeout);
        // Only after a timeout: wait (bounded) for this CTA's copies still in
        // flight before its shared memory goes away.
        int qq = q;
        uint32_t pp = parity;
        for (int64_t lj = li; lj < nlocal && lj < li + nstage; ++lj) {
            (void)mbar_wait_bounded(smem_addr(&sbar[qq]), pp);
            if (++qq == nstage) {
                qq = 0;
                pp ^= 1u;
            }
        }
    }
    cl.sync();     // no CTA leaves while another may still push into its slots
}

// ---------------------------------------------------------------------------
// host-side planning and launch
// ---------------------------------------------------------------------------

inline int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }
inline int round_up32(int v) { return (v + 31) & ~31; }

// Raises a kernel's dynamic shared memory limit to the device's opt-in
// maximum less the kernel's static shared memory (needed above 48 KB, before
// occupancy queries and launches).
inline cudaError_t allow_smem(const void *fn, const LaunchCtx &ctx, int bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                ctx.smem_optin - (int)fa.sharedSizeBytes);
}

// The shifted kernel's form with per-column copies (CS) for chain C and vpt
// slots, with the staged ring when stg, or nullptr: defined and instantiated
// in the rows_shift_cs_*.cu units only.  In a chain's own unit those kernels changed how ptxas allocated that
// unit's other kernels (the two-slot staged bf16 LayerNorm kernel went from 32
// registers and an 8-byte stack to 38 registers: three 512-thread CTAs an SM
// instead of four).
template <class C> const void *shift_cs_fn(int vpt, bool stg);
// The cluster kernel's form for rows off the 16-byte grid (SH) for chain C,
// vpt slots, staged or not, on a launch of `threads` threads, or nullptr:
// defined and instantiated in the rows_cluster_sh_*.cu units only, for the
// same reason.
template <class C> const void *cluster_sh_fn(int vpt, bool staged, int threads);

template <class C> struct RowEngine {
    using T = typename C::T;
    static constexpr int kVecN = C::kVec;     // elements per vector slot

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
    // A kernel's launch bound and whether it spills beyond `tolerance` bytes.
    static mb_status kernel_limits(const void *f, int *max_threads, bool *spills,
                                   size_t tolerance = kSpillTolerance) {
        cudaFuncAttributes fa;
        const cudaError_t e = cudaFuncGetAttributes(&fa, f);
        if (e != cudaSuccess) return cuda_fail(e);
        *max_threads = fa.maxThreadsPerBlock;
        *spills = fa.localSizeBytes > tolerance;
        return MB_OK;
    }
    // Threads per CTA of the one-warp-per-row engine: with at most
    // kWarpBlock / 32 rows per SM, one CTA per SM holding ceil(rows / SMs)
    // warps, so every SM gets the same rows at once; else kWarpBlock-thread
    // CTAs.  Measured on GB300 (graph, steady state): the 1024 x 1024
    // Inductor chain 2.95 us on 147 CTAs of 7 warps against 2.99 on 512 CTAs
    // of 2 (bf16 2.33 against 2.37).
    static int warp_threads(const LaunchCtx &ctx, int64_t rows) {
        const int64_t per_sm = (rows + ctx.sm_count - 1) / ctx.sm_count;
        return per_sm >= kWarpBlock / 32 ? kWarpBlock : 32 * (int)(per_sm > 0 ? per_sm : 1);
    }
    // Longest row (in vector slots) one CTA holds.
    static int cta_max_nvec(bool vec) {
        return vec ? kCtaMaxThreads * max_vpt(true)
                   : (max_vpt(false) >= C::kWideScalarSlots ? kWideThreads : kCtaMaxThreads) *
                         max_vpt(false);
    }
    // The CTA engine's kernels: the register-capped form for chains that ask
    // for it (C::kRegCap) on the staged vector shapes it was measured on (one
    // or two slots; elsewhere the cap spills), the 512-thread form for the
    // scalar slot counts that spill under the 1024-thread bound
    // (C::kWideScalarSlots and up), the ordinary one otherwise.
    template <int VPT, int VEC, bool STAGED> static const void *cta_kernel() {
        if constexpr (C::kRegCap && STAGED && VEC == kVecN && VPT <= 2)
            return (const void *)rows_cta_kernel_capped<C, VPT, VEC, STAGED>;
        else if constexpr (VEC == 1 && VPT >= C::kWideScalarSlots)
            return (const void *)rows_cta_kernel_wide<C, VPT, VEC, STAGED>;
        else return (const void *)rows_cta_kernel<C, VPT, VEC, STAGED>;
    }
    static const void *cta_fn(int vpt, bool vec, bool staged) {
        if (vec) {
            if (staged) {
                switch (vpt) {
                    case 1: return cta_kernel<1, kVecN, true>();
                    case 2: return cta_kernel<2, kVecN, true>();
                    case 4: return cta_kernel<4, kVecN, true>();
                    case 8: if constexpr (kVecN == 4) return cta_kernel<8, kVecN, true>();
                            break;
                }
            } else {
                switch (vpt) {
                    case 1: return cta_kernel<1, kVecN, false>();
                    case 2: return cta_kernel<2, kVecN, false>();
                    case 4: return cta_kernel<4, kVecN, false>();
                    case 8: if constexpr (kVecN == 4) return cta_kernel<8, kVecN, false>();
                            break;
                }
            }
        } else if (!staged) {
            switch (vpt) {
                case 1: return cta_kernel<1, 1, false>();
                case 2: return cta_kernel<2, 1, false>();
                case 4: return cta_kernel<4, 1, false>();
                case 8: return cta_kernel<8, 1, false>();
                case 16: return cta_kernel<16, 1, false>();
                case 32: return cta_kernel<32, 1, false>();
            }
        }
        return nullptr;
    }

    // The shifted-vector kernel (rows off the 16-byte grid), vpt vector slots;
    // cs: per-column arrays copied to shared memory (chains that have some),
    // stg: with them, the rows' vectors staged by bulk copies.
    static const void *shift_fn(int vpt, bool cs, bool stg = false) {
        if constexpr (C::kShiftOk) {
            if constexpr (C::kColArrays > 0 || C::kShiftStaged) {
                if (cs) return shift_cs_fn<C>(vpt, stg);
            }
            switch (vpt) {
                case 1: return (const void *)rows_shift_kernel<C, 1>;
                case 2: return (const void *)rows_shift_kernel<C, 2>;
                case 4: return (const void *)rows_shift_kernel<C, 4>;
                case 8: if constexpr (kVecN == 4) return (const void *)rows_shift_kernel<C, 8>;
                        break;
            }
        }
        return nullptr;
    }
    // Shared memory of the shifted kernel's per-column copies (its CS form),
    // and of one stage of its ring (STG: the row inputs' whole vectors).
    static int64_t shift_col_bytes(int cols) {
        return (int64_t)C::kColArrays * (((int64_t)cols + 15) & ~(int64_t)15) * (int64_t)sizeof(T);
    }
    static int64_t shift_stage_bytes(int cols) {
        return (int64_t)C::kInputs * (((int64_t)cols + 15) & ~(int64_t)15) * (int64_t)sizeof(T);
    }

    // The cluster kernel for a launch of `threads` threads: the 512-thread
    // form for 32 or more values per thread when the CTA fits it, else the
    // 1024-thread form.
    template <int VPT, int VEC, bool STAGED> static const void *cluster_kernel(int threads) {
        if constexpr (VPT * VEC >= 32) {
            if (threads <= kWideThreads)
                return (const void *)rows_cluster_kernel<C, VPT, VEC, STAGED, kWideThreads>;
        }
        return (const void *)rows_cluster_kernel<C, VPT, VEC, STAGED, kCtaMaxThreads>;
    }
    static const void *cluster_fn(int vpt, bool vec, bool staged, int threads, bool sh = false) {
        if constexpr (C::kShiftOk && !C::kPartialRows) {
            if (sh) return cluster_sh_fn<C>(vpt, staged, threads);
        }
        if (sh) return nullptr;
        if (vec) {
            if (staged) {
                switch (vpt) {
                    case 1: return cluster_kernel<1, kVecN, true>(threads);
                    case 2: return cluster_kernel<2, kVecN, true>(threads);
                    case 4: return cluster_kernel<4, kVecN, true>(threads);
                    case 8: if constexpr (kVecN == 4) return cluster_kernel<8, kVecN, true>(threads);
                            break;
                }
            } else {
                switch (vpt) {
                    case 1: return cluster_kernel<1, kVecN, false>(threads);
                    case 2: return cluster_kernel<2, kVecN, false>(threads);
                    case 4: return cluster_kernel<4, kVecN, false>(threads);
                    case 8: if constexpr (kVecN == 4) return cluster_kernel<8, kVecN, false>(threads);
                            break;
                }
            }
        } else if (!staged) {
            switch (vpt) {
                case 1: return cluster_kernel<1, 1, false>(threads);
                case 2: return cluster_kernel<2, 1, false>(threads);
                case 4: return cluster_kernel<4, 1, false>(threads);
                case 8: return cluster_kernel<8, 1, false>(threads);
                case 16: return cluster_kernel<16, 1, false>(threads);
                case 32: return cluster_kernel<32, 1, false>(threads);
            }
        }
        return nullptr;
    }

    // Resident clusters of `fn` with `cs` CTAs of `threads` threads (0 if none fit).
    static mb_status active_clusters(const LaunchCtx &ctx, const void *fn, int cs, int threads,
                                     int smem, int *n) {
        cudaError_t e = cudaSuccess;
        if (cs > 8)
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess) e = allow_smem(fn, ctx, smem);
        if (e != cudaSuccess) return cuda_fail(e);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs * ctx.sm_count);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = (size_t)smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(n, fn, &cfg);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();   // an unplaceable shape is not an error here
            *n = 0;
        }
        return MB_OK;
    }

    // One cluster of `cs` CTAs per row.  Each resident cluster keeps one row
    // in flight, so among cluster sizes 2, 4, 8, 16 (or the requested one) and
    // the vectors-per-thread that fit a slice in one CTA, take the launch with
    // the most resident clusters (ties: the smaller cluster, then the more
    // values per thread); no rank is empty.  Launches holding at most the
    // chain's C::kClusterVals values per thread come first: a thread keeps
    // its slice and the next row's prefetch in registers.
    // sh: rows off the 16-byte grid on the cluster kernel's SH form (nvec:
    // the most whole vectors any row has).
    static mb_status plan_cluster(const LaunchCtx &ctx, const RowTuning &tun, int64_t rows,
                                  int nvec, bool vec, RowPlan *p, const void **fn,
                                  bool sh = false) {
        const int VEC = vec ? kVecN : 1;
        for (int pass = 0; pass < 2; ++pass) {
            mb_status st = plan_cluster_pass(ctx, tun, rows, nvec, vec,
                                             pass == 0 ? C::kClusterVals / VEC : 1 << 30, p, fn,
                                             sh);
            if (st != MB_ERR_SHAPE) return st;
        }
        return MB_ERR_SHAPE;
    }

    // The shared-memory-resident cluster kernel (bf16 rows of chains with
    // C::kStageLargeSlices): among cluster sizes 2, 4, 8, 16 (or the
    // requested one) whose CTA slice is kClusterStageMin bytes or more, the
    // most resident clusters (ties: the smaller cluster), a ring of two
    // stages where it fits (or the requested depth).  MB_ERR_SHAPE when no
    // slice is that large (the register kernels serve those rows).  Sweeps on
    // GB300, softmax bf16 (µs, register-staged against this kernel): 65536
    // columns 446 / 399, 131072 534 / 437, 262144 601 / 462, 524288 695 /
    // 566; with 32 and 40 KB slices (32776, 40000 columns) the register
    // kernels stay ahead.
    static mb_status plan_cluster_smem(const LaunchCtx &ctx, const RowTuning &tun, int64_t rows,
                                       int nvec, RowPlan *p, const void **fn) {
        const void *f = (const void *)rows_cluster_smem_kernel<C, kVecN>;
        int bn = 0, bcs = 0, bthr = 0, bslice = 0, bring = 0, bsmem = 0;
        for (int cs0 : {2, 4, 8, 16}) {
            int cs = cs0;
            if (tun.stages >= 2 && tun.stages <= kMaxCluster) {
                if (cs0 != 2) continue;
                cs = tun.stages;
            }
            if (cs > nvec) cs = nvec;
            const int slice_v = ceil_div(nvec, cs);
            cs = ceil_div(nvec, slice_v);                  // no empty rank
            if (cs < 2) continue;
            const int64_t sb = (int64_t)C::kInputs * slice_v * kVecN * (int64_t)sizeof(T);
            if (sb < kClusterStageMin || sb + kHdrBytes > ctx.smem_optin) continue;
            int ring = tun.ctas_per_sm > 0 ? tun.ctas_per_sm : 2;
            if (ring > kMaxStages) ring = kMaxStages;
            while (ring > 1 && ring * sb + kHdrBytes > ctx.smem_optin) --ring;
            const int threads = slice_v < kCtaMaxThreads ? round_up32(slice_v) : kCtaMaxThreads;
            int n = 0;
            mb_status st = active_clusters(ctx, f, cs, threads, (int)(ring * sb), &n);
            if (st != MB_OK) return st;
            if (n > bn) {
                bn = n; bcs = cs; bthr = threads; bslice = slice_v; bring = ring;
                bsmem = (int)(ring * sb);
            }
        }
        if (!bn) return MB_ERR_SHAPE;
        *fn = f;
        const int64_t ncl = rows < bn ? rows : bn;
        p->path = MB_ROW_CLUSTER; p->threads = bthr; p->vpt = ceil_div(bslice, bthr);
        p->stages = bcs; p->smem = bsmem;
        p->ctas = (int)(ncl * bcs);
        p->slice = bslice;
        p->ring = bring;
        p->cap = bn;
        return MB_OK;
    }

    static mb_status plan_cluster_pass(const LaunchCtx &ctx, const RowTuning &tun,
                                       int64_t rows, int nvec, bool vec, int max_vpt_regs,
                                       RowPlan *p, const void **fn, bool sh) {
        // Staged (bulk-async ring) for bf16 rows that are vectorised and in
        // device memory, ring depth kClusterRing; fp32 rows load directly,
        // except for chains that ask (C::kStageLargeSlices) when a CTA's slice
        // is at least kClusterStageMin bytes, ring depth 2.  Sweeps on GB300:
        // LN at 65536 columns, bf16 staged 4.24 TB/s against 3.49 direct (its
        // register prefetch holds unpacked floats, halving the resident
        // threads), fp32 direct 6.10 against 5.53 staged; fp32 softmax staged
        // 6.0-6.7 against 5.0-6.3 direct for slices of 64 KB and more (65536
        // to 524288 columns), direct ahead for smaller ones.  A requested
        // depth (ctas_per_sm on this path) stages any dtype.
        const bool may_stage = vec && !tun.no_bulk;
        const bool staged = may_stage && (sizeof(T) == 2 || tun.ctas_per_sm > 0);
        if constexpr (C::kStageLargeSlices && sizeof(T) == 2) {
            if (staged && !sh) {
                const mb_status st = plan_cluster_smem(ctx, tun, rows, nvec, p, fn);
                if (st != MB_ERR_SHAPE) return st;
            }
        }
        const int VEC = vec ? kVecN : 1;
        int best_n = 0, best_cs = 0, best_vpt = 0, best_threads = 0, best_slice = 0;
        int best_ring = 0, best_smem = 0;
        bool best_spills = true;
        for (int cs0 : {2, 4, 8, 16}) {
            int cs = cs0;
            if (tun.stages >= 2 && tun.stages <= kMaxCluster) {
                if (cs0 != 2) continue;
                cs = tun.stages;
            }
            if (cs > nvec) cs = nvec;
            const int slice_v = ceil_div(nvec, cs);
            cs = ceil_div(nvec, slice_v);                  // no empty rank
            if (cs < 2) continue;
            const int64_t stage_bytes = (int64_t)C::kInputs * slice_v * VEC * (int64_t)sizeof(T);
            int ring = 0, smem = 0;
            const bool stage_f32 = may_stage && C::kStageLargeSlices && sizeof(T) == 4 &&
                                   stage_bytes >= kClusterStageMin;
            if (staged || stage_f32) {
                ring = tun.ctas_per_sm > 0 ? tun.ctas_per_sm : (staged ? kClusterRing : 2);
                if (ring > kMaxStages) ring = kMaxStages;
                // (the kernel's static shared memory stays within kHdrBytes)
                while (ring > 1 && ring * stage_bytes + kHdrBytes > ctx.smem_optin) --ring;
                if (stage_bytes + kHdrBytes > ctx.smem_optin) ring = 0;   // direct loads
                smem = (int)(ring * stage_bytes);
            }
            for (int vpt = 1; vpt <= max_vpt(vec); vpt *= 2) {
                if (tun.vpt > 0 && vpt != tun.vpt) continue;
                if (tun.vpt <= 0 && vpt > max_vpt_regs) continue;
                // the first pass leaves out the 1024-thread form of the
                // 32-value kernels (it spills); the second takes it when
                // nothing else fits (fp32 rows of 524288)
                if (tun.vpt <= 0 && max_vpt_regs < (1 << 30) && vpt * VEC >= 32 &&
                    ceil_div(slice_v, vpt) > kWideThreads)
                    continue;
                if (ceil_div(slice_v, vpt) > kCtaMaxThreads) continue;
                const int threads = round_up32(ceil_div(slice_v, vpt));
                const void *f = cluster_fn(vpt, vec, ring > 0, threads, sh);
                if (!f) continue;
                int max_threads = 0;
                bool spills = false;
                mb_status st = kernel_limits(f, &max_threads, &spills);
                if (st != MB_OK) return st;
                if (threads > max_threads) continue;    // the kernel's launch bound
                int n = 0;
                st = active_clusters(ctx, f, cs, threads, smem, &n);
                if (st != MB_OK) return st;
                // a spilling kernel only when no other serves; ties keep the
                // smaller cluster (fewer exchange partners), and within it the
                // more values per thread (fewer, busier threads)
                const bool better =
                    n > 0 && (best_n == 0 || (best_spills && !spills) ||
                              (spills == best_spills &&
                               (n > best_n || (n == best_n && cs == best_cs))));
                if (better) {
                    best_n = n; best_cs = cs; best_vpt = vpt; best_threads = threads;
                    best_slice = slice_v; best_ring = ring; best_smem = smem;
                    best_spills = spills;
                }
            }
        }
        if (!best_n && tun.vpt > 0) {
            RowTuning t2 = tun;
            t2.vpt = 0;
            return plan_cluster(ctx, t2, rows, nvec, vec, p, fn, sh);
        }
        if (!best_n) return MB_ERR_SHAPE;       // the caller tries the next pass
        *fn = cluster_fn(best_vpt, vec, best_ring > 0, best_threads, sh);
        const int64_t ncl = rows < best_n ? rows : best_n;
        p->shift = sh ? 1 : 0;
        p->path = MB_ROW_CLUSTER; p->threads = best_threads; p->vpt = best_vpt;
        p->stages = best_cs; p->smem = best_smem;
        p->ctas = (int)(ncl * best_cs);
        p->slice = best_slice;
        p->ring = best_ring;
        p->cap = best_n;
        return MB_OK;
    }

    // CTAs of `fn` resident per SM with `threads` threads and `smem` bytes.
    static mb_status occupancy(const LaunchCtx &ctx, const void *fn, int threads, int smem,
                               int *occ) {
        cudaError_t e = allow_smem(fn, ctx, smem);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fn, threads, smem);
        if (e != cudaSuccess) return cuda_fail(e);
        return MB_OK;
    }

    // The occupancy-derived part of a plan depends on the device, the row
    // length, the alignment and the tuning, not on the row count: it is
    // computed once (for an unbounded row count) and kept here; each call
    // only sizes the grid for its rows.
    struct CacheEntry {
        bool used;
        int device, cols, aligned, path, ctas_per_sm, stages, vpt, no_bulk, outs, read_pct;
        RowPlan core;
        const void *fn;
    };
    static constexpr int kCacheSize = 64;
    struct PlanCache {
        std::mutex mu;
        CacheEntry entries[kCacheSize] = {};
        int next = 0;
    };
    static PlanCache &plan_cache() {
        static PlanCache c;      // one per chain type, built on first use
        return c;
    }

    // The one-CTA engines' grid for `rows` rows on `cap` resident CTAs.
    // Balanced: as many row rounds as the full grid needs, but only as many
    // CTAs as those rounds need, so the last round is not mostly idle (8192
    // rows on 608 slots: 14 rounds on 586 CTAs, not 13.5 on 608).  With the
    // shifted kernel's per-column copies (cs), a multiple of the period of
    // the rows' offsets within 16 bytes where the cap allows, so that each CTA
    // meets one offset and makes its copy once (the cap, SMs x CTAs per SM,
    // is a multiple of 8 on 152 SMs; elsewhere the copy is redone as a CTA's
    // offset changes).
    static int64_t cta_grid(int64_t rows, int64_t cap, int cols, bool cs) {
        int64_t grid = rows < cap ? rows : cap;
        if (grid > 0) {
            const int64_t rounds = (rows + grid - 1) / grid;
            grid = (rows + rounds - 1) / rounds;
        }
        if (cs && rows > grid) {
            const int64_t step = ((int64_t)cols * (int64_t)sizeof(T)) & 15;
            int64_t period = 1;
            while ((step * period) & 15) period *= 2;
            const int64_t up = (grid + period - 1) / period * period;
            if (grid > period && up <= cap) grid = up;
        }
        return grid;
    }

    static mb_status plan(const LaunchCtx &ctx, const RowTuning &tun, int64_t rows, int cols,
                          int aligned, RowPlan *p, const void **fn) {
        RowPlan core;
        const void *f = nullptr;
        bool hit = false;
        PlanCache &pc = plan_cache();
        {
            std::lock_guard<std::mutex> lock(pc.mu);
            for (const CacheEntry &e : pc.entries) {
                if (e.used && e.device == ctx.device && e.cols == cols && e.aligned == (int)aligned &&
                    e.path == tun.path && e.ctas_per_sm == tun.ctas_per_sm &&
                    e.stages == tun.stages && e.vpt == tun.vpt && e.no_bulk == tun.no_bulk &&
                    e.outs == tun.outs && e.read_pct == tun.read_pct) {
                    core = e.core;
                    f = e.fn;
                    hit = true;
                    break;
                }
            }
        }
        if (!hit) {
            mb_status st = plan_full(ctx, tun, kUnboundedRows, cols, aligned, &core, &f);
            if (st != MB_OK) return st;
            std::lock_guard<std::mutex> lock(pc.mu);
            pc.entries[pc.next] = CacheEntry{true, ctx.device, cols, (int)aligned, tun.path,
                                             tun.ctas_per_sm, tun.stages, tun.vpt, tun.no_bulk,
                                             tun.outs, tun.read_pct, core, f};
            pc.next = (pc.next + 1) % kCacheSize;
        }
        *p = core;
        *fn = f;
        if (core.path == MB_ROW_WARP) {
            const int threads = warp_threads(ctx, rows);
            const int64_t cap = core.cap * (kWarpBlock / threads);
            const int64_t want = (rows + threads / 32 - 1) / (threads / 32);
            p->threads = threads;
            p->ctas = (int)(want < cap ? want : cap);
        } else if (core.path == MB_ROW_CLUSTER) {
            const int64_t ncl = rows < core.cap ? rows : core.cap;
            p->ctas = (int)(ncl * core.stages);
        } else {
            if (core.shift >= 2 && rows <= core.cap1) {
                // one row per CTA: copying the per-column values would cost
                // as much as reading them once, so the kernel without copies
                *fn = shift_fn(core.vpt, false);
                p->path = MB_ROW_DIRECT;
                p->shift = 1;
                p->smem = kHdrBytes;
                p->stages = 0;
            }
            p->ctas = (int)cta_grid(rows, core.cap, cols, p->shift >= 2);
        }
        return MB_OK;
    }

    // `aligned`: 1 every pointer of the call is 16-byte aligned; 2 every row
    // tensor (inputs and outputs) starts at the same offset within 16 bytes,
    // the per-column vectors anywhere; 0 neither.
    static mb_status plan_full(const LaunchCtx &ctx, const RowTuning &tun, int64_t rows, int cols,
                               int aligned, RowPlan *p, const void **fn) {
        const bool vec = aligned == 1 && (cols % kVecN) == 0;
        // rows off the 16-byte grid whose tensors share their offset within
        // 16 bytes: shifted vectors on one CTA (at least one whole vector a row)
        const bool shift_ok = !vec && aligned >= 1 && C::kShiftOk && cols >= 2 * kVecN;
        const int VEC = vec ? kVecN : 1;
        const int nvec = cols / VEC;
        const int nvec_shift = ceil_div(cols, kVecN);      // a row's vector slots, at most
        const bool warp_ok = nvec <= 32 * 8;
        const int stage_bytes = C::kInputs * cols * (int)sizeof(T);
        const bool stage_fits = !tun.no_bulk && kHdrBytes + stage_bytes <= ctx.smem_optin;

        const bool shift = shift_ok && nvec_shift <= cta_max_nvec(true);
        const bool one_cta = shift || nvec <= cta_max_nvec(vec);
        int warp_vpl = 1;
        while (warp_vpl * 32 < nvec) warp_vpl *= 2;
        bool warp_spills = false;
        if (warp_ok) {
            int max_threads = 0;
            mb_status st = kernel_limits(warp_fn(warp_vpl, vec), &max_threads, &warp_spills);
            if (st != MB_OK) return st;
        }
        int path = tun.path;
        if (path == MB_ROW_WARP && !warp_ok) path = MB_ROW_AUTO;
        if (path == MB_ROW_STAGED && (!vec || !stage_fits || !one_cta)) path = MB_ROW_AUTO;
        if (path == MB_ROW_DIRECT && !one_cta) path = MB_ROW_AUTO;
        if (path == MB_ROW_CLUSTER && nvec < 2) path = MB_ROW_AUTO;
        // one warp per row unless its kernel for this length spills (the
        // dropout chains' longest warp rows); then one CTA per row
        if (path == MB_ROW_AUTO)
            path = !one_cta ? MB_ROW_CLUSTER
                 : warp_ok && !warp_spills ? MB_ROW_WARP
                 : (vec && stage_fits ? MB_ROW_STAGED : MB_ROW_DIRECT);

        p->vec = VEC;
        if (path == MB_ROW_CLUSTER) {
            // rows off the 16-byte grid with a common offset: the cluster
            // kernel's shifted form, on the most whole vectors a row has
            if (shift_ok && !C::kPartialRows) {
                p->vec = kVecN;
                return plan_cluster(ctx, tun, rows, cols / kVecN, true, p, fn, true);
            }
            return plan_cluster(ctx, tun, rows, nvec, vec, p, fn);
        }
        if (path == MB_ROW_WARP) {
            const int vpl = warp_vpl;
            *fn = warp_fn(vpl, vec);
            int occ = 0;
            mb_status st = occupancy(ctx, *fn, kWarpBlock, 0, &occ);
            if (st != MB_OK) return st;
            if (tun.ctas_per_sm > 0 && tun.ctas_per_sm < occ) occ = tun.ctas_per_sm;
            if (occ < 1) occ = 1;
            p->cap = (int64_t)occ * ctx.sm_count;
            const int threads = warp_threads(ctx, rows);
            occ *= kWarpBlock / threads;
            const int64_t want = (rows + threads / 32 - 1) / (threads / 32);
            const int64_t cap = (int64_t)occ * ctx.sm_count;
            p->path = path; p->threads = threads; p->vpt = vpl; p->stages = 0; p->smem = 0;
            p->ctas = (int)(want < cap ? want : cap);
            return MB_OK;
        }

        // CTA engine.  Each resident CTA keeps one row in flight, so pick the
        // vectors-per-thread that lets the most CTAs share an SM, counting up
        // to a target, then the most threads per SM; one ring stage counted
        // for the staged path.  The target is the per-SM byte budget over one
        // row's reads and writes (on the staged path reads count over the
        // share of the row the chain reads: a causal score row's copy holds
        // its unmasked prefix only),
        // rounded to the nearest row count between 2 and kMaxRowsInFlight,
        // unless the chain sets its own; the grid holds no more resident CTAs
        // than the target.
        const bool staged = path == MB_ROW_STAGED;
        const bool shifted = shift && path == MB_ROW_DIRECT;
        const int nvec_cta = shifted ? nvec_shift : nvec;
        // Shifted rows may take the kernel's shared-memory forms: cstage, the
        // copies of the chain's per-column arrays (when they fit one CTA), and
        // sstaged, with them a ring streaming the rows' vectors (when one stage
        // fits beside the copies, for chains that take it, and not when the
        // direct path is asked for).  A chain without per-column arrays (the
        // row softmax) has the ring alone, or neither.  The choice among the
        // forms that fit is made below.
        bool cstage = shifted && (C::kColArrays > 0 || C::kShiftStaged) && !tun.no_bulk &&
                      kHdrBytes + shift_col_bytes(cols) <= ctx.smem_optin;
        bool sstaged = cstage && C::kShiftStaged && tun.path != MB_ROW_DIRECT &&
                       kHdrBytes + shift_col_bytes(cols) + shift_stage_bytes(cols) <= ctx.smem_optin;
        if (C::kColArrays == 0 && !sstaged) cstage = false;
        const int64_t row_io =
            ((int64_t)C::kInputs * cols * (staged ? tun.read_pct : 100) / 100 +
             (int64_t)tun.outs * cols) *
            (int64_t)sizeof(T);
        // The shifted kernel loads its rows straight into registers; with two
        // row inputs its fp32 rows keep HBM busy only from the bf16 budget on
        // (sweeps on GB300, LayerNorm + residual rows of 2051 to 8195 fp32
        // values: fastest at 8, 5, 4, 3 and 2 rows an SM).
        const int64_t budget = sizeof(T) == 2 || (shifted && C::kInputs == 2)
                                   ? kFlightBytesBf16 : kFlightBytesF32;
        int64_t want_rows = row_io > 0 ? (budget + row_io / 2) / row_io : kMaxRowsInFlight;
        if (want_rows > kMaxRowsInFlight) want_rows = kMaxRowsInFlight;
        int target = want_rows < 2 ? 2 : (int)want_rows;
        if (C::kRowsTarget > 0) target = C::kRowsTarget;     // the chain's own measured target
        struct Pick {
            int vpt = 0, occ = 0, threads = 0;
            bool spills = true;
        };
        auto pick = [&](bool cs, bool stg, Pick &best) -> mb_status {
            const int smem_q = kHdrBytes + (staged ? stage_bytes : 0) +
                               (cs ? (int)shift_col_bytes(cols) : 0) +
                               (stg ? (int)shift_stage_bytes(cols) : 0);
            for (int cand = 1; cand <= max_vpt(vec || shifted); cand *= 2) {
                if (tun.vpt > 0 && cand != tun.vpt) continue;
                if (ceil_div(nvec_cta, cand) > kCtaMaxThreads) continue;
                const int threads = round_up32(ceil_div(nvec_cta, cand));
                // shifted rows: no CTA of fewer than four warps where the row
                // allows more (LayerNorm + residual, fp32 rows of 2051: eight
                // CTAs of 96 threads an SM ran 13% slower than five of 288)
                if (shifted && threads < 128 && nvec_cta >= 128) continue;
                const void *f = shifted ? shift_fn(cand, cs, stg) : cta_fn(cand, vec, staged);
                if (!f) continue;
                int max_threads = 0;
                bool spills = false;
                mb_status st = kernel_limits(f, &max_threads, &spills,
                                             shifted ? kShiftSpillTolerance : kSpillTolerance);
                if (st != MB_OK) return st;
                if (threads > max_threads) continue;          // the kernel's launch bound
                int occ = 0;
                st = occupancy(ctx, f, threads, smem_q, &occ);
                if (st != MB_OK) return st;
                if (tun.ctas_per_sm > 0 && tun.ctas_per_sm < occ) occ = tun.ctas_per_sm;
                if (occ < 1) continue;
                const int rows_in_flight = occ < target ? occ : target;
                const int best_rows = best.occ < target ? best.occ : target;
                // a spilling kernel only when no other serves; then the most
                // rows in flight, tie-broken on threads per SM, counting the
                // CTAs that will be resident once the target caps them
                const bool better =
                    best.vpt == 0 || (best.spills && !spills) ||
                    (spills == best.spills &&
                     (rows_in_flight > best_rows ||
                      (rows_in_flight == best_rows &&
                       rows_in_flight * threads > best_rows * best.threads)));
                if (better) best = Pick{cand, occ, threads, spills};
            }
            return MB_OK;
        };
        // Shifted rows: the staged form where it fits, unless it spills where
        // the copies alone do not (a staged CTA keeps a second row in flight
        // in its ring, so it is not judged by its CTAs an SM: LN fp32 4099
        // columns ran 82.2 us staged at three CTAs an SM against 86.9 with
        // the copies alone at four); else the copies alone, or neither when
        // that keeps more rows in flight or spills less (the copies take
        // shared memory: w and b of an fp32 row of 16383, 128 KB a CTA).
        Pick best;
        mb_status pst = pick(cstage, sstaged, best);
        if (pst != MB_OK) return pst;
        auto wins = [&](const Pick &c, const Pick &b) {
            const int rb_ = b.occ < target ? b.occ : target;
            const int rc_ = c.occ < target ? c.occ : target;
            return c.vpt && (!b.vpt || (b.spills && !c.spills) || (b.spills == c.spills && rc_ > rb_));
        };
        if (sstaged) {
            // the copies alone, or (no per-column arrays) the plain form
            const bool next_cs = C::kColArrays > 0;
            Pick next;
            if ((pst = pick(next_cs, false, next)) != MB_OK) return pst;
            if (next.vpt && (!best.vpt || (best.spills && !next.spills))) {
                best = next;
                sstaged = false;
                cstage = next_cs;
            }
        }
        if (cstage && !sstaged) {
            Pick plain;
            if ((pst = pick(false, false, plain)) != MB_OK) return pst;
            if (wins(plain, best)) {
                best = plain;
                cstage = false;
                sstaged = false;
            }
        }
        int best_vpt = best.vpt, best_occ = best.occ, best_threads = best.threads;
        if (tun.ctas_per_sm <= 0 && best_occ > target) best_occ = target;
        if (!best_vpt && tun.vpt > 0) {
            RowTuning t2 = tun;
            t2.vpt = 0;
            return plan(ctx, t2, rows, cols, aligned, p, fn);
        }
        if (!best_vpt) return MB_ERR_SHAPE;

        int stages = 0, smem = kHdrBytes, occ = best_occ;
        if (staged) {
            // One stage per CTA when several CTAs share an SM (their rows
            // overlap one another); two when a CTA is alone.  A requested
            // depth is honoured as far as shared memory allows.
            int want = tun.stages > 0 ? tun.stages : (best_occ >= 2 ? 1 : 2);
            if (want > kMaxStages) want = kMaxStages;
            while (want > 1 && (int64_t)occ * (kHdrBytes + 1024 + (int64_t)want * stage_bytes) >
                                   ctx.smem_per_sm)
                --want;
            while (want > 1 && kHdrBytes + (int64_t)want * stage_bytes > ctx.smem_optin) --want;
            stages = want;
            smem = kHdrBytes + stages * stage_bytes;
        }
        *fn = shifted ? shift_fn(best_vpt, cstage, sstaged) : cta_fn(best_vpt, vec, staged);
        if (shifted) { p->vec = kVecN; p->shift = 1; }
        if (cstage) { smem = kHdrBytes + (int)shift_col_bytes(cols); p->shift = 2; }
        if (sstaged) {
            // the staged path's ring depth rule, beside the copies
            const int64_t sb = shift_stage_bytes(cols);
            int want = tun.stages > 0 ? tun.stages : (best_occ >= 2 ? 1 : 2);
            if (want > kMaxStages) want = kMaxStages;
            while (want > 1 && (int64_t)occ * (smem + 1024 + want * sb) > ctx.smem_per_sm) --want;
            while (want > 1 && smem + want * sb > ctx.smem_optin) --want;
            stages = want;
            smem += (int)(want * sb);
            p->shift = 3;
        }
        int occ2 = 0;
        mb_status st = occupancy(ctx, *fn, best_threads, smem, &occ2);
        if (st != MB_OK) return st;
        if (occ2 < occ) occ = occ2;
        if (occ < 1) occ = 1;
        const int64_t cap = (int64_t)occ * ctx.sm_count;
        p->cap = cap;
        if (cstage) {
            // a launch of one row per CTA skips the copies (plan() below)
            int occ1 = 0;
            st = occupancy(ctx, shift_fn(best_vpt, false), best_threads, kHdrBytes, &occ1);
            if (st != MB_OK) return st;
            p->cap1 = (int64_t)(occ1 < occ ? occ1 : occ) * ctx.sm_count;
        }
        p->path = sstaged ? MB_ROW_STAGED : path;
        p->threads = best_threads; p->vpt = best_vpt; p->stages = stages;
        p->smem = smem;
        p->ctas = (int)cta_grid(rows, cap, cols, p->shift >= 2);
        return MB_OK;
    }

    static mb_status run(const LaunchCtx &ctx, const RowTuning &tun, const typename C::Args &a,
                         int64_t rows, int cols, int aligned, RowPlan *plan_out, bool launch) {
        RowPlan p;
        const void *fn = nullptr;
        RowTuning tn = tun;      // the per-call planning inputs
        if (C::outputs(a) > tn.outs) tn.outs = C::outputs(a);
        tn.read_pct = C::read_percent(a, rows, cols);
        mb_status st = plan(ctx, tn, rows, cols, aligned, &p, &fn);
        if (st != MB_OK) return st;
        if (launch &&
            (p.path == MB_ROW_STAGED || (p.path == MB_ROW_CLUSTER && p.ring > 0) || p.shift >= 2)) {
            // Asynchronous copies into shared memory are planned for device
            // memory only: rows (bulk copies) or per-column arrays (the
            // shifted kernel's copies) held in host memory (pinned, read over
            // the host link) take a plain-load path.
            bool dev = true;
            if (p.shift >= 2) {
                for (int i = 0; i < C::kColArrays; ++i) dev = dev && device_resident(C::col_array(a, i));
            }
            if (p.shift != 2) {
                for (int i = 0; i < C::kInputs; ++i) dev = dev && device_resident(a.in[i]);
            }
            if (!dev) {
                RowTuning t2 = tn;
                t2.no_bulk = 1;
                if ((st = plan(ctx, t2, rows, cols, aligned, &p, &fn)) != MB_OK) return st;
            }
        }
        if (plan_out) *plan_out = p;
        if (!launch || rows == 0) return MB_OK;
        LaunchCtx lctx = ctx;
        lctx.pdl = ctx.pdl && rows * cols * (int64_t)sizeof(T) * (C::kInputs + 1) <= kOverlapMaxBytes;
        typename C::Args args = a;
        int64_t rows_arg = rows;
        int cols_arg = cols;
        // the fourth kernel argument: ring depth, the cluster's slice length,
        // or (shifted vectors) the row tensors' common offset within 16 bytes,
        // with the ring depth above it on the staged shifted form
        int stages_arg = p.path == MB_ROW_CLUSTER ? p.slice * p.vec
                       : p.shift ? (int)(reinterpret_cast<uintptr_t>(a.in[0]) & 15u) |
                                       (p.shift == 3 ? p.stages << 8 : 0)
                       : (p.stages > 0 ? p.stages : 1);
        unsigned *err = ctx.dev_err;
        // the cluster kernel's sixth argument: the ring depth, with (shifted
        // rows) the row tensors' common offset within 16 bytes above it
        int ring_arg = p.ring | (p.path == MB_ROW_CLUSTER && p.shift
                                     ? (int)(reinterpret_cast<uintptr_t>(a.in[0]) & 15u) << 8
                                     : 0);
        void *kargs[] = {&args, &rows_arg, &cols_arg, &stages_arg, &err, &ring_arg};
        cudaError_t e = launch_kernel(lctx, fn, dim3(p.ctas), dim3(p.threads), kargs, p.smem,
                                      p.path == MB_ROW_CLUSTER ? p.stages : 1);
        if (e != cudaSuccess) return cuda_fail(e);
        return MB_OK;
    }
};

}  // namespace mb
