// Instantiations of the compact-output router forward, staged path:
// softmax score, f32 logits.
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_staged_compact_softmax_f32(const FwdArgs& a, const StagedPlan& p, int* status,
                                           cudaStream_t st) {
  return launch_staged<SF_SOFTMAX, DT_F32, 2>(a, p, status, st);
}
int occupancy_staged_compact_softmax_f32(const StagedPlan& p) {
  return staged_occupancy<SF_SOFTMAX, DT_F32, 2>(p);
}
}  // namespace moe_router
