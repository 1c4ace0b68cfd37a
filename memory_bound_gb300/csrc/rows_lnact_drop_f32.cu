// rows_lnact_drop_f32.cu -- LayerNorm family (optional residual, residual-stream
// output, activation none / relu / gelu-tanh, optional per-row statistics),
// fp32 I/O, with dropout on the activation output.
#include "lnact_run.cuh"

namespace mb {

mb_status lnact_drop_rows_f32(const LaunchCtx &ctx, const RowTuning &tun, bool residual,
                              const void *x, const void *r, const void *w, const void *b, void *out,
                              void *h, int64_t rows, int cols, float eps, int act, const LnExtras &ex,
                              int aligned, RowPlan *plan, bool launch) {
    return lnact_run<float, true>(ctx, tun, residual, x, r, w, b, out, h, rows, cols, eps, act,
                                ex, aligned, plan, launch);
}

}  // namespace mb
