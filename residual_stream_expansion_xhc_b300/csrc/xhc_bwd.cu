// Backward of the xHC sublayer update, small passes (bf16 state):
//   W^T prep     the bf16 K-major copy of W used by the tensor-core stream pass
//   reduce       fixed-order sums of the weight-gradient partials
// The column pass and the per-token reverse are in xhc_stream.cu, the
// tensor-core stream pass (dX for every stream, dW) in xhc_tc.cu.
//
// Method: "xHC: Expanded Hyper-Connections" (qingkeai.online), sections
// "Scaling N" (H^pre/H^post/H^res, Sinkhorn), "Temporal Feature Augmentation"
// (causal depthwise convolutions 4/8/12), "Dense read, sparse write" (only the
// k active streams are written).
#include <algorithm>

#include "xhc_bwd.cuh"

namespace xhc {

// ============================================================== W^T in bf16
//
// Wt[col][q] = bf16(W[q][col]) for q < P, zero for P <= q < 64: the K-major
// operand of dV = dP . W in the stream pass, as a hi part and a lo part
// (Wt + NC * 64 holds bf16(W - hi)), so that hi + lo keeps about 16 bits of W.

__global__ void wt_prep_kernel(const float* __restrict__ W, __nv_bfloat16* __restrict__ Wt, int P, size_t NC) {
  __shared__ float tile[64][65];
  const size_t col0 = (size_t)blockIdx.x * 64;
  for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) {
    const int q = i / 64, c = i % 64;
    tile[q][c] = (q < P && col0 + c < NC) ? W[(size_t)q * NC + col0 + c] : 0.0f;
  }
  __syncthreads();
  __nv_bfloat16* Wt_lo = Wt + NC * 64;
  for (int i = threadIdx.x; i < 64 * 32; i += blockDim.x) {
    const int c = i / 32, q2 = (i % 32) * 2;
    if (col0 + c < NC) {
      const float a = tile[q2][c], b = tile[q2 + 1][c];
      const uint32_t h = pack_bf2(a, b);
      *reinterpret_cast<uint32_t*>(Wt + (col0 + c) * 64 + q2) = h;
      *reinterpret_cast<uint32_t*>(Wt_lo + (col0 + c) * 64 + q2) = pack_bf2(a - bf_lo(h), b - bf_hi(h));
    }
  }
}

// Fixed-order sums: conv-weight partials [rows][24][C] and dW partials
// [ranges][P][N C].
__global__ void bwd_reduce_kernel(int conv_rows, int C, const float* __restrict__ cpart, float* __restrict__ dw4,
                                  float* __restrict__ dw8, float* __restrict__ dw12, int w_ranges, size_t PNC,
                                  const float* __restrict__ wpart, float* __restrict__ dW) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (cpart) {
    for (size_t i = i0; i < (size_t)NTAPS * C; i += stride) {
      const int g = (int)(i / C), c = (int)(i % C);
      // eight independent loads in flight, then a fixed-order sum
      float s = 0.0f;
      int r = 0;
      for (; r + 8 <= conv_rows; r += 8) {
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = cpart[((size_t)(r + q) * NTAPS + g) * C + c];
#pragma unroll
        for (int q = 0; q < 8; ++q) s += v[q];
      }
      for (; r < conv_rows; ++r) s += cpart[((size_t)r * NTAPS + g) * C + c];
      if (g < 4) dw4[(size_t)c * 4 + g] = s;
      else if (g < 12) dw8[(size_t)c * 8 + (g - 4)] = s;
      else dw12[(size_t)c * 12 + (g - 12)] = s;
    }
  }
  for (size_t i = i0; i < PNC; i += stride) {
    float s = 0.0f;
    for (int r = 0; r < w_ranges; ++r) s += wpart[(size_t)r * PNC + i];
    dW[i] = s;
  }
}

// ============================================================== launchers

cudaError_t launch_wt_prep(const Params& p, const float* W, __nv_bfloat16* Wt, cudaStream_t st) {
  const size_t NC = (size_t)p.N * p.C;
  timing_begin("bwd_wt_prep", st);
  wt_prep_kernel<<<(unsigned)((NC + 63) / 64), 256, 0, st>>>(W, Wt, p.P, NC);
  timing_end(st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_reduce(const Params& p, const BwdArgs<__nv_bfloat16>& a, bool has_conv, const float* cpart,
                              int conv_rows, int w_ranges, const float* wpart, cudaStream_t st) {
  const size_t PNC = (size_t)p.P * p.N * p.C;
  timing_begin("bwd_reduce", st);
  bwd_reduce_kernel<<<592, 256, 0, st>>>(conv_rows, p.C, has_conv ? cpart : nullptr, a.dw[0],
                                         a.dw[1], a.dw[2], w_ranges, PNC, wpart, a.dW);
  timing_end(st);
  return cudaGetLastError();
}

}  // namespace xhc
