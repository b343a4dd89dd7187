// tcgen05 chunk attention (bf16, head_dim 128, page 128) -- placeholder until the
// tensor-core kernels land; every shape runs the SIMT kernels meanwhile.
#include "attn_common.cuh"

namespace oomb {

bool tc_supported(const Geometry& g) {
  (void)g;
  return false;
}

cudaError_t launch_attn_fwd_tc(const AttnArgs& a, cudaStream_t st) { return launch_attn_fwd_simt(a, st); }
cudaError_t launch_attn_bwd_tc(const AttnArgs& a, cudaStream_t st) { return launch_attn_bwd_simt(a, st); }

}  // namespace oomb
