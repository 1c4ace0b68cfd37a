// rows_inductor_bf16.cu -- the TorchInductor example chain with bf16 I/O
// (inputs widened exactly, fp32 steps, y rounded once).
#include "chains.cuh"

namespace mb {

mb_status inductor_rows_bf16(const LaunchCtx &ctx, const RowTuning &tun, const void *x,
                             const void *bias, const void *gamma, const void *beta, void *y,
                             int64_t rows, int cols, float x_scale, float branch_scale,
                             int aligned, RowPlan *plan, bool launch) {
    using C = InductorChainT<uint16_t>;
    C::Args a{{static_cast<const uint16_t *>(x)}, static_cast<const uint16_t *>(bias),
              static_cast<const uint16_t *>(gamma), static_cast<const uint16_t *>(beta),
              static_cast<uint16_t *>(y), x_scale, branch_scale};
    return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
}

}  // namespace mb
