// Instantiations of the router backwards (top-K and aux scores).
#include "router_launch.cuh"

namespace moe_router {
cudaError_t launch_bwd_any(int sf, int dt, const BwdArgs& a, const BwdConfig& c,
                           cudaStream_t st) {
  if (sf == SF_SOFTMAX) {
    return dt == DT_F32 ? launch_bwd<SF_SOFTMAX, DT_F32>(a, c, st)
                        : launch_bwd<SF_SOFTMAX, DT_BF16>(a, c, st);
  }
  if (sf == SF_SOFTMAX_POST) {
    return dt == DT_F32 ? launch_bwd<SF_SOFTMAX_POST, DT_F32>(a, c, st)
                        : launch_bwd<SF_SOFTMAX_POST, DT_BF16>(a, c, st);
  }
  return dt == DT_F32 ? launch_bwd<SF_SIGMOID, DT_F32>(a, c, st)
                      : launch_bwd<SF_SIGMOID, DT_BF16>(a, c, st);
}
}  // namespace moe_router
