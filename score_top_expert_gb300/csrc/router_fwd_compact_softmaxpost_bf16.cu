// Instantiations of the compact-output router forward, segment path:
// post-softmax score, bf16 logits.
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_fwd_compact_softmaxpost_bf16(const FwdArgs& a, const FwdConfig& c, cudaStream_t st) {
  return launch_fwd<SF_SOFTMAX_POST, DT_BF16, 2>(a, c, st);
}
}  // namespace moe_router
