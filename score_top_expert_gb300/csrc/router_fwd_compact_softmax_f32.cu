// Instantiations of the compact-output router forward, segment path:
// softmax score, f32 logits.
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_fwd_compact_softmax_f32(const FwdArgs& a, const FwdConfig& c, cudaStream_t st) {
  return launch_fwd<SF_SOFTMAX, DT_F32, 2>(a, c, st);
}
}  // namespace moe_router
