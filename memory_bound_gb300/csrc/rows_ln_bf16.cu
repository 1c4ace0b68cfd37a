// rows_ln_bf16.cu -- residual + LayerNorm + GeLU-tanh, bf16 I/O, fp32 math.
#include "chains.cuh"

namespace mb {

mb_status ln_gelu_rows_bf16(const LaunchCtx &ctx, const RowTuning &tun, const void *x,
                            const void *r, const void *w, const void *b, void *out,
                            int64_t rows, int cols, float eps, int aligned, RowPlan *plan,
                            bool launch) {
    using C = LnGeluChain<uint16_t>;
    C::Args a{{static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(r)},
              static_cast<const uint16_t *>(w), static_cast<const uint16_t *>(b),
              static_cast<uint16_t *>(out), eps, 1.0f / (float)cols};
    return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
}

}  // namespace mb
