// Instantiations of the fused decode router with expert maps (segment path):
// softmax score, bf16 logits.
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_fwd_maps_softmax_bf16(const FwdArgs& a, const FwdConfig& c, cudaStream_t st) {
  return launch_fwd<SF_SOFTMAX, DT_BF16, 3>(a, c, st);
}
}  // namespace moe_router
