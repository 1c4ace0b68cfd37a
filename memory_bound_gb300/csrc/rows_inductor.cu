// rows_inductor.cu -- the TorchInductor example chain (bias, relu, branches,
// row mean, affine epilogue), fp32.
#include "chains.cuh"

namespace mb {

mb_status inductor_rows_f32(const LaunchCtx &ctx, const RowTuning &tun, const float *x,
                            const float *bias, const float *gamma, const float *beta,
                            float *y, int64_t rows, int cols, float x_scale,
                            float branch_scale, int aligned, RowPlan *plan, bool launch) {
    using C = InductorChain;
    C::Args a{{x}, bias, gamma, beta, y, x_scale, branch_scale};
    return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
}

}  // namespace mb
