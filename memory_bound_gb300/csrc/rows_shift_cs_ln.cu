// rows_shift_cs_ln.cu -- shifted rows with per-column copies: residual +
// LayerNorm + GeLU and the TorchInductor chain, fp32 and bf16.
#include "rows_shift_cs.cuh"

namespace mb {

template const void *shift_cs_fn<LnGeluChain<float>>(int, bool);
template const void *shift_cs_fn<LnGeluChain<uint16_t>>(int, bool);
template const void *shift_cs_fn<InductorChainT<float>>(int, bool);
template const void *shift_cs_fn<InductorChainT<uint16_t>>(int, bool);

}  // namespace mb
