// Instantiations of the fused decode router with expert maps (staged path,
// one block): post-softmax score, bf16 logits.
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_staged_maps_softmaxpost_bf16(const FwdArgs& a, const StagedPlan& p, int* status,
                                        cudaStream_t st) {
  return launch_staged<SF_SOFTMAX_POST, DT_BF16, 3>(a, p, status, st);
}
int occupancy_staged_maps_softmaxpost_bf16(const StagedPlan& p) {
  return staged_occupancy<SF_SOFTMAX_POST, DT_BF16, 3>(p);
}
}  // namespace moe_router
