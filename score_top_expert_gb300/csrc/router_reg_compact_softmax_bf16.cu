// Instantiations of the register-resident router forward with compact
// outputs: softmax score, bf16 logits.
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_reg_compact_softmax_bf16(const FwdArgs& a, const RegPlan& p, int* status,
                                            cudaStream_t st) {
  return reg_dispatch<SF_SOFTMAX, DT_BF16, false, 2>(a, p, status, st, nullptr);
}
int occupancy_reg_compact_softmax_bf16(const RegPlan& p) {
  int n = 0;
  reg_dispatch<SF_SOFTMAX, DT_BF16, true, 2>(FwdArgs{}, p, nullptr, nullptr, &n);
  return n;
}
}  // namespace moe_router
