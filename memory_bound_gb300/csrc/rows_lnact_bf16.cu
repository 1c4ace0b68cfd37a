// rows_lnact_bf16.cu -- LayerNorm family (optional residual, residual-stream
// output, activation none / relu / gelu-tanh, optional per-row statistics),
// bf16 I/O, without dropout.
#include "lnact_run.cuh"

namespace mb {

mb_status lnact_rows_bf16(const LaunchCtx &ctx, const RowTuning &tun, bool residual,
                          const void *x, const void *r, const void *w, const void *b, void *out,
                          void *h, int64_t rows, int cols, float eps, int act, const LnExtras &ex,
                          int aligned, RowPlan *plan, bool launch) {
    return lnact_run<uint16_t, false>(ctx, tun, residual, x, r, w, b, out, h, rows, cols, eps, act,
                                ex, aligned, plan, launch);
}

}  // namespace mb
