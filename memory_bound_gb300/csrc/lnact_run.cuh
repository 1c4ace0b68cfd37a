// lnact_run.cuh -- builds the LayerNorm family's kernel arguments (with the
// optional statistics and dropout) and runs the row engine; each
// rows_lnact*.cu instantiates it for one I/O type, with or without dropout.
#pragma once

#include <cmath>

#include "chains.cuh"

namespace mb {

// The dropout launch constants for probability p and key (seed, offset): the
// Philox key schedule written out, the integer keep threshold and the scale.
inline DropoutArgs make_dropout(float p, uint64_t seed, uint64_t offset) {
    DropoutArgs d{};
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        d.rk[2 * r] = k0;
        d.rk[2 * r + 1] = k1;
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
    d.offset = offset;
    // keep iff half * 2^-16 >= p  <=>  half >= ceil(p * 2^16) (p * 2^16 is
    // exact; a threshold of 2^16 keeps nothing)
    d.thr = (uint32_t)std::ceil((double)p * 65536.0);
    d.inv_keep = 1.0f / (1.0f - p);
    return d;
}

template <typename T, bool DROP>
mb_status lnact_run(const LaunchCtx &ctx, const RowTuning &tun, bool residual, const void *x,
                    const void *r, const void *w, const void *b, void *out, void *h,
                    int64_t rows, int cols, float eps, int act, const LnExtras &ex,
                    int aligned, RowPlan *plan, bool launch) {
    auto fill = [&](auto &a) {
        a.w = static_cast<const T *>(w);
        a.b = static_cast<const T *>(b);
        a.out = static_cast<T *>(out);
        a.h = static_cast<T *>(h);
        a.eps = eps;
        a.inv_cols = 1.0f / (float)cols;
        a.act = act;
        a.mean_out = ex.mean;
        a.rstd_out = ex.rstd;
        if constexpr (DROP) a.drop = make_dropout(ex.p, ex.seed, ex.offset);
    };
    if (residual) {
        using C = LnActChain<T, true, DROP>;
        typename C::Args a{};
        a.in[0] = static_cast<const T *>(x);
        a.in[1] = static_cast<const T *>(r);
        fill(a);
        return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
    }
    using C = LnActChain<T, false, DROP>;
    typename C::Args a{};
    a.in[0] = static_cast<const T *>(x);
    fill(a);
    return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
}

}  // namespace mb
