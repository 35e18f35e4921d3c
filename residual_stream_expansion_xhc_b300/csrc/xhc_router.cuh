// Router with per-token active sets (bf16 state, see xhc_router.cu).
#pragma once

#include "xhc_kernels.cuh"

namespace xhc {

// W' [P, N*C] for the router's projection pass: rows 0 .. N-1 = W_r, row N = 1
// (the projection then gives the sum of the state), the other rows 0; and the
// row sums rs [N] of W_r (fixed order).
cudaError_t launch_router_weights(const Params& p, const float* W_r, float* Wp, float* rs, cudaStream_t st);

// Per token from the router pass's logits zr [T, P+1] (rstd-scaled W' v, then
// rstd): LayerNorm scores s = sigmoid(r), r = W_r LN(v), the active slots (the
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

}  // namespace xhc
