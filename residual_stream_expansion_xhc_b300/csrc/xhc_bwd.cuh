// Backward passes of the xHC update for bf16 state (see xhc_bwd.cu, xhc_tc.cu).
#pragma once

#include "xhc_kernels.cuh"

namespace xhc {

cudaError_t launch_wt_prep(const Params& p, const float* W, __nv_bfloat16* Wt, cudaStream_t st);
// W^T (as launch_wt_prep; with W_r non-NULL its N rows follow W's P rows) and
// the coefficient block from saved logits (as launch_coef) in one launch.
cudaError_t launch_bwd_prep(const Params& p, const float* W, const float* W_r, __nv_bfloat16* Wt,
                            const float* saved, float* coef, cudaStream_t st);
// Fixed-order sums of the conv-weight partials [conv_rows][24][C] and the dW
// partials [w_ranges][P][N C].
// With a router (dW_r non-NULL) the dW partials have P + N rows; the W_r rows
// go to dW_r less c_r = sum_t cm[t] (computed here into c_r [N]).
cudaError_t launch_bwd_reduce(const Params& p, const BwdArgs<__nv_bfloat16>& a, bool has_conv, const float* cpart,
                              int conv_rows, int w_ranges, const float* wpart, cudaStream_t st,
                              float* dW_r = nullptr, const float* cm = nullptr, float* c_r = nullptr);

// Token ranges the tensor-core stream pass splits the batch into (each range
// writes one dW partial).
int bwd_stream_ranges(const Params& p);
cudaError_t launch_bwd_stream_tc(const Params& p, const BwdArgs<__nv_bfloat16>& a, const __nv_bfloat16* Wt,
                                 const __nv_bfloat16* dP, int ranges, float* wpart, cudaStream_t st);

// H^res logits from the active rows: full projection from W_pp, W_ra; and
// the gradient of W_ra from the full dW (C a multiple of 4).
cudaError_t launch_hres_active_weights(const Params& p, const float* W_pp, const float* W_ra, float* W,
                                       cudaStream_t st);
cudaError_t launch_hres_active_grad(const Params& p, const float* dW, float* dW_ra, cudaStream_t st);

}  // namespace xhc
