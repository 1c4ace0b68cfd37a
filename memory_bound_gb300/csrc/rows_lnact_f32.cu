// rows_lnact_f32.cu -- LayerNorm family (optional residual, residual-stream
// output, activation none / relu / gelu-tanh), fp32 I/O.
#include "chains.cuh"

namespace mb {

mb_status lnact_rows_f32(const LaunchCtx &ctx, const RowTuning &tun, bool residual,
                         const void *x, const void *r, const void *w, const void *b, void *out,
                         void *h, int64_t rows, int cols, float eps, int act, bool aligned,
                         RowPlan *plan, bool launch) {
    using T = float;
    const T *px = static_cast<const T *>(x), *pr = static_cast<const T *>(r);
    const T *pw = static_cast<const T *>(w), *pb = static_cast<const T *>(b);
    T *po = static_cast<T *>(out), *ph = static_cast<T *>(h);
    if (residual) {
        using C = LnActChain<T, true>;
        C::Args a{{px, pr}, pw, pb, po, ph, eps, act};
        return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
    }
    using C = LnActChain<T, false>;
    C::Args a{{px}, pw, pb, po, ph, eps, act};
    return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
}

}  // namespace mb
