// rows_cluster_sh_ln.cu -- rows longer than a CTA and off the 16-byte grid:
// residual + LayerNorm + GeLU and the TorchInductor chain, fp32 and bf16.
#include "rows_cluster_sh.cuh"

namespace mb {

template const void *cluster_sh_fn<LnGeluChain<float>>(int, bool, int);
template const void *cluster_sh_fn<LnGeluChain<uint16_t>>(int, bool, int);
template const void *cluster_sh_fn<InductorChainT<float>>(int, bool, int);
template const void *cluster_sh_fn<InductorChainT<uint16_t>>(int, bool, int);

}  // namespace mb
