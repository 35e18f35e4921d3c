// Router with per-token active sets (bf16 state, see xhc_router.cu).
#pragma once

#include "xhc_kernels.cuh"

namespace xhc {

// Per token from the router's record inputs zr [T, P+1] (rstd W_r v at
// 0..N-1, rstd sum(v) at N, rstd at P; launch_coeffs_tc_router): LayerNorm scores s = sigmoid(r), r = W_r LN(v), the active slots (the
// nf fixed streams, then the top k - nf others by score) into `tok_idx`
// [T, k], and the router record rrec [T, 2N+2] = (s, r, LN mean, LN sd); the
// coefficient block's H^post rows of the routed slots are scaled by their
// scores.
cudaError_t launch_route(const Params& p, const float* zr, const float* rs, const int32_t* fixed, int nf,
                         int32_t* tok_idx, float* rrec, float* coef, cudaStream_t st);

// Backward helpers: the routed slots' H^post rows scaled by their scores
// (from tok_idx and the router record), and the row sums of W_r.
cudaError_t launch_route_scale(const Params& p, const int32_t* tok_idx, const float* rrec, int nf, float* coef,
                               cudaStream_t st);
cudaError_t launch_router_rowsums(const Params& p, const float* W_r, float* rs, cudaStream_t st);

// The state before an in-place routed update from the state after it: the
// saved old active rows saved_active [T, k, C] (bf16) written back into
// X [T, N, C] at each token's slots tok_idx [T, k].
cudaError_t launch_restore_active(const Params& p, void* X, const void* saved_active, const int32_t* tok_idx, int sms,
                                  cudaStream_t st);

}  // namespace xhc
