// rows_softmax.cu -- row softmax, fp32 or bf16 I/O (fp32 arithmetic).
#include "chains.cuh"

namespace mb {

mb_status softmax_rows(const LaunchCtx &ctx, const RowTuning &tun, mb_dtype dtype,
                       const void *x, void *y, int64_t rows, int cols, int aligned,
                       RowPlan *plan, bool launch) {
    if (dtype == MB_F32) {
        using C = SoftmaxChain<float>;
        C::Args a{{static_cast<const float *>(x)}, static_cast<float *>(y)};
        return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
    }
    using C = SoftmaxChain<uint16_t>;
    C::Args a{{static_cast<const uint16_t *>(x)}, static_cast<uint16_t *>(y)};
    return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
}

}  // namespace mb
