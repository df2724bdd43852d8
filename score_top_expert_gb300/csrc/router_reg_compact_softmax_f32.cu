// Instantiations of the register-resident router forward with compact
// outputs: softmax score, f32 logits.
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_reg_compact_softmax_f32(const FwdArgs& a, const RegPlan& p, int* status,
                                           cudaStream_t st) {
  return reg_dispatch<SF_SOFTMAX, DT_F32, false, 2>(a, p, status, st, nullptr);
}
int occupancy_reg_compact_softmax_f32(const RegPlan& p) {
  int n = 0;
  reg_dispatch<SF_SOFTMAX, DT_F32, true, 2>(FwdArgs{}, p, nullptr, nullptr, &n);
  return n;
}
}  // namespace moe_router
