// tcgen05 chunk-attention backward (bf16, head_dim 128, page 128).
#include "tc_common.cuh"

namespace oomb {

cudaError_t launch_attn_bwd_tc(const AttnArgs& a, cudaStream_t st) { return launch_attn_bwd_simt(a, st); }

}  // namespace oomb
