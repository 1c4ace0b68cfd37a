// rows_shift_cs_softmax.cu -- shifted rows of the row softmax on the staged
// ring (the chain has no per-column arrays to copy), bf16.
#include "rows_shift_cs.cuh"

namespace mb {

template const void *shift_cs_fn<SoftmaxChain<uint16_t>>(int, bool);

}  // namespace mb
