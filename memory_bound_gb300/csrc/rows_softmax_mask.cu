// rows_softmax_mask.cu -- softmax of attention-score rows: scaled, with an
// optional causal mask; fp32 or bf16 I/O (fp32 arithmetic).
#include "chains.cuh"

namespace mb {

mb_status softmax_mask_rows(const LaunchCtx &ctx, const RowTuning &tun, mb_dtype dtype,
                            const void *x, void *y, int64_t rows, int cols, float scale,
                            bool causal, int64_t period, int64_t offset, int aligned,
                            RowPlan *plan, bool launch) {
    if (period < 1) period = 1;
    if (offset > cols) offset = cols;                 // masks nothing more
    const uint64_t recip = ~0ull / (uint64_t)period;
    if (dtype == MB_F32) {
        using C = ScaleMaskSoftmaxChain<float>;
        C::Args a{{static_cast<const float *>(x)}, static_cast<float *>(y), scale, causal ? 1 : 0,
                  period, offset, recip};
        return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
    }
    using C = ScaleMaskSoftmaxChain<uint16_t>;
    C::Args a{{static_cast<const uint16_t *>(x)}, static_cast<uint16_t *>(y), scale,
              causal ? 1 : 0, period, offset, recip};
    return RowEngine<C>::run(ctx, tun, a, rows, cols, aligned, plan, launch);
}

}  // namespace mb
