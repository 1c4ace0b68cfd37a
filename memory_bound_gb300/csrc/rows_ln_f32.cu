// rows_ln_f32.cu -- residual + LayerNorm + GeLU-tanh, fp32 I/O.
#include "chains.cuh"

namespace mb {

mb_status ln_gelu_rows_f32(const LaunchCtx &ctx, const RowTuning &tun, const void *x,
                           const void *r, const void *w, const void *b, void *out,
                           int64_t rows, int cols, float eps, int aligned, RowPlan *plan,
                           bool launch) {
    using C = LnGeluChain<float>;
    C::Args a{{static_cast<const float *>(x), static_cast<const float *>(r)},
              static_cast<const float *>(w), static_cast<const float *>(b),
              static_cast<float *>(out), eps, 1.0f / (float)cols};
    return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
}

}  // namespace mb
