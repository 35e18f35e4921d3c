// Backward passes of the xHC update for bf16 state (see xhc_bwd.cu, xhc_tc.cu).
#pragma once

#include "xhc_kernels.cuh"

namespace xhc {

// Rows of conv-weight partial sums written by the TFA pass.
size_t bwd_conv_partial_rows(const Params& p);

cudaError_t launch_wt_prep(const Params& p, const float* W, __nv_bfloat16* Wt, cudaStream_t st);
cudaError_t launch_bwd_token(const Params& p, const BwdArgs<__nv_bfloat16>& a, bool has_conv, __nv_bfloat16* dP,
                             cudaStream_t st);
cudaError_t launch_bwd_tfa(const Params& p, const BwdArgs<__nv_bfloat16>& a, bool has_conv, float* cpart,
                           cudaStream_t st);
cudaError_t launch_bwd_reduce(const Params& p, const BwdArgs<__nv_bfloat16>& a, bool has_conv, const float* cpart,
                              int w_ranges, const float* wpart, cudaStream_t st);

// Token ranges the tensor-core stream pass splits the batch into (each range
// writes one dW partial).
int bwd_stream_ranges(const Params& p);
cudaError_t launch_bwd_stream_tc(const Params& p, const BwdArgs<__nv_bfloat16>& a, const __nv_bfloat16* Wt,
                                 const __nv_bfloat16* dP, int ranges, float* wpart, cudaStream_t st);

}  // namespace xhc
