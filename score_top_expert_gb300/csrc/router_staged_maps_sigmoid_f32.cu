// Instantiations of the fused decode router with expert maps (staged path,
// one block): sigmoid score, f32 logits.
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_staged_maps_sigmoid_f32(const FwdArgs& a, const StagedPlan& p, int* status,
                                        cudaStream_t st) {
  return launch_staged<SF_SIGMOID, DT_F32, 3>(a, p, status, st);
}
int occupancy_staged_maps_sigmoid_f32(const StagedPlan& p) {
  return staged_occupancy<SF_SIGMOID, DT_F32, 3>(p);
}
}  // namespace moe_router
