// Instantiations of the router forwards: post-softmax score, f32 logits.
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_fwd_softmaxpost_f32(const FwdArgs& a, const FwdConfig& c, cudaStream_t st) {
  return launch_fwd<SF_SOFTMAX_POST, DT_F32>(a, c, st);
}
}  // namespace moe_router
