// rows_cluster_sh_softmax.cu -- rows longer than a CTA and off the 16-byte
// grid: the row softmax, fp32 and bf16.
#include "rows_cluster_sh.cuh"

namespace mb {

template const void *cluster_sh_fn<SoftmaxChain<float>>(int, bool, int);
template const void *cluster_sh_fn<SoftmaxChain<uint16_t>>(int, bool, int);

}  // namespace mb
