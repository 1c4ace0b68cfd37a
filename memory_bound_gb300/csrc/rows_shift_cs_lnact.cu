// rows_shift_cs_lnact.cu -- shifted rows with per-column copies: the
// LayerNorm family without dropout (with and without a residual), fp32 and
// bf16.
#include "rows_shift_cs.cuh"

namespace mb {

template const void *shift_cs_fn<LnActChain<float, false, false>>(int, bool);
template const void *shift_cs_fn<LnActChain<float, true, false>>(int, bool);
template const void *shift_cs_fn<LnActChain<uint16_t, false, false>>(int, bool);
template const void *shift_cs_fn<LnActChain<uint16_t, true, false>>(int, bool);

}  // namespace mb
