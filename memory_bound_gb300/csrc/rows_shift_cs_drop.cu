// rows_shift_cs_drop.cu -- shifted rows with per-column copies: the
// LayerNorm family with dropout (with and without a residual), fp32 and bf16.
#include "rows_shift_cs.cuh"

namespace mb {

template const void *shift_cs_fn<LnActChain<float, false, true>>(int, bool);
template const void *shift_cs_fn<LnActChain<float, true, true>>(int, bool);
template const void *shift_cs_fn<LnActChain<uint16_t, false, true>>(int, bool);
template const void *shift_cs_fn<LnActChain<uint16_t, true, true>>(int, bool);

}  // namespace mb
