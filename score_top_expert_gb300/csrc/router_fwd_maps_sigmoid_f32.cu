// Instantiations of the fused decode router with expert maps (segment path):
// sigmoid score, f32 logits.
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_fwd_maps_sigmoid_f32(const FwdArgs& a, const FwdConfig& c, cudaStream_t st) {
  return launch_fwd<SF_SIGMOID, DT_F32, 3>(a, c, st);
}
}  // namespace moe_router
