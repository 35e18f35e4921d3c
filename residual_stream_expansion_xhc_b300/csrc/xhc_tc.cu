// Tensor-core kernels of the xHC update (sm_103a).
#include "xhc_tc.cuh"

namespace xhc {

bool tc_coeffs_supported(const Params&) { return false; }
cudaError_t launch_coeffs_tc(const Params&, const void*, const float*, float*, float*, float*, float*, void*,
                             cudaStream_t) {
  return cudaErrorNotSupported;
}
bool tc_update_supported(const Params&) { return false; }
cudaError_t launch_update_tc(const Params&, const UpdArgs<__nv_bfloat16>&, bool, cudaStream_t) {
  return cudaErrorNotSupported;
}
bool tc_bwd_supported(const Params&) { return false; }
size_t tc_bwd_partial_bytes(const Params&) { return 0; }
cudaError_t launch_bwd_tc(const Params&, const BwdArgs<__nv_bfloat16>&, bool, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace xhc
