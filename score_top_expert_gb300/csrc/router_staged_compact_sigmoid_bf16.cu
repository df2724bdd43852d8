// Instantiations of the compact-output router forward, staged path:
// sigmoid score, bf16 logits.
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_staged_compact_sigmoid_bf16(const FwdArgs& a, const StagedPlan& p, int* status,
                                           cudaStream_t st) {
  return launch_staged<SF_SIGMOID, DT_BF16, 2>(a, p, status, st);
}
int occupancy_staged_compact_sigmoid_bf16(const StagedPlan& p) {
  return staged_occupancy<SF_SIGMOID, DT_BF16, 2>(p);
}
}  // namespace moe_router
