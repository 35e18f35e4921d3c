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

// With a router, entries P .. P + R - 1 carry W_r^T (R = N router rows).
__device__ __forceinline__ void wt_prep_block(const float* __restrict__ W, const float* __restrict__ W_r, int R,
                                              __nv_bfloat16* __restrict__ Wt, int P, size_t NC, size_t blk) {
  __shared__ float tile[64][65];
  const size_t col0 = blk * 64;
  for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) {
    const int q = i / 64, c = i % 64;
    float v = 0.0f;
    if (col0 + c < NC) {
      if (q < P) v = W[(size_t)q * NC + col0 + c];
      else if (W_r && q < P + R) v = W_r[(size_t)(q - P) * NC + col0 + c];
    }
    tile[q][c] = v;
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

__global__ void __launch_bounds__(256) wt_prep_kernel(const float* __restrict__ W, __nv_bfloat16* __restrict__ Wt,
                                                      int P, size_t NC) {
  wt_prep_block(W, nullptr, 0, Wt, P, NC, blockIdx.x);
}

// The two independent preparations of the backward in one launch: blocks
// [0, nwt) build W^T, the others the coefficient block from the saved logits.
__global__ void __launch_bounds__(256) bwd_prep_kernel(Params p, const float* __restrict__ W,
                                                       const float* __restrict__ W_r,
                                                       __nv_bfloat16* __restrict__ Wt, unsigned nwt,
                                                       const float* __restrict__ saved, float* __restrict__ coef,
                                                       size_t T_all) {
  if (blockIdx.x < nwt) wt_prep_block(W, W_r, p.N, Wt, p.P, (size_t)p.N * p.C, blockIdx.x);
  else coef_block(p, saved, coef, T_all, blockIdx.x - nwt);
}

// Fixed-order sums: conv-weight partials [rows][24][C] and dW partials
// [ranges][P][N C].  The first `cblocks` blocks take the conv-weight sums,
// the others the dW sums, four consecutive entries (one 16-byte vector) per
// thread and step.
// With a router each range's partial has the N rows of W_r after W's P rows
// (PNC covers both, RNC0 = P N C is where they start): they go to dW_r, less
// the LayerNorm mean term c_r[row] (the same for every column of a row).
__global__ void bwd_reduce_kernel(int conv_rows, int C, const float* __restrict__ cpart, float* __restrict__ dw4,
                                  float* __restrict__ dw8, float* __restrict__ dw12, int cblocks, int w_ranges,
                                  size_t PNC, const float* __restrict__ wpart, float* __restrict__ dW,
                                  size_t RNC0, size_t NC, float* __restrict__ dW_r, const float* __restrict__ c_r) {
  if ((int)blockIdx.x < cblocks) {
    const size_t stride = (size_t)cblocks * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)NTAPS * C; i += stride) {
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
    return;
  }
  // PNC is a multiple of 4 (C is a multiple of 8) and the buffers are 16-byte aligned
  const size_t n4 = PNC / 4;
  const size_t stride = (size_t)(gridDim.x - cblocks) * blockDim.x;
  const float4* wp = reinterpret_cast<const float4*>(wpart);
  for (size_t i = (size_t)(blockIdx.x - cblocks) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 s = wp[i];
    for (int r = 1; r < w_ranges; ++r) {
      const float4 v = wp[(size_t)r * n4 + i];
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    if (4 * i < RNC0) {
      reinterpret_cast<float4*>(dW)[i] = s;
    } else {
      const size_t j = 4 * i - RNC0;
      const float c = c_r[j / NC];
      reinterpret_cast<float4*>(dW_r)[j / 4] = make_float4(s.x - c, s.y - c, s.z - c, s.w - c);
    }
  }
}

// c_r[n] = sum over tokens of cm[t][n]: one block per n, fixed-order sums.
__global__ void __launch_bounds__(256) column_sum_kernel(const float* __restrict__ cm, size_t T_all, int N,
                                                         float* __restrict__ out) {
  __shared__ float part[256];
  float s = 0.0f;
  for (size_t t = threadIdx.x; t < T_all; t += 256) s += cm[t * N + blockIdx.x];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) part[threadIdx.x] += part[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) out[blockIdx.x] = part[0];
}

// ============================================================== H^res from the active rows
//
// Section "Dense read, sparse write": the mixing logits generated from the k
// active streams only.  The full projection W [P, N*C] carries W_ra in the
// active streams' columns of its H^res rows (zeros elsewhere); the gradient
// of W_ra is read back from the same columns.  One thread per 4 columns.

__global__ void hres_active_weights_kernel(Params p, const float* __restrict__ W_pp, const float* __restrict__ W_ra,
                                           float* __restrict__ W) {
  const size_t NC = (size_t)p.N * p.C;
  const size_t n4 = (size_t)p.P * NC / 4;
  const int R0 = p.N + 4 * p.k;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = (4 * i) / NC, col = (4 * i) % NC;
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if ((int)r < R0) {
      v = *reinterpret_cast<const float4*>(W_pp + r * NC + col);
    } else {
      const int n = (int)(col / p.C), c = (int)(col % p.C), slot = p.is_active[n];
      if (slot) v = *reinterpret_cast<const float4*>(W_ra + (r - R0) * ((size_t)p.k * p.C) + (size_t)(slot - 1) * p.C + c);
    }
    *reinterpret_cast<float4*>(W + r * NC + col) = v;
  }
}

__global__ void hres_active_grad_kernel(Params p, const float* __restrict__ dW, float* __restrict__ dW_ra) {
  const size_t kC = (size_t)p.k * p.C;
  const size_t n4 = (size_t)p.k * p.k * kC / 4;
  const size_t NC = (size_t)p.N * p.C;
  const int R0 = p.N + 4 * p.k;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const size_t q = (4 * i) / kC, col = (4 * i) % kC;
    const int j = (int)(col / p.C), c = (int)(col % p.C);
    *reinterpret_cast<float4*>(dW_ra + q * kC + col) =
        *reinterpret_cast<const float4*>(dW + (R0 + q) * NC + (size_t)p.idx[j] * p.C + c);
  }
}

cudaError_t launch_hres_active_weights(const Params& p, const float* W_pp, const float* W_ra, float* W,
                                       cudaStream_t st) {
  const size_t n4 = (size_t)p.P * p.N * p.C / 4;
  const unsigned grid = (unsigned)std::min<size_t>((n4 + 255) / 256, 148 * 16);
  hres_active_weights_kernel<<<grid, 256, 0, st>>>(p, W_pp, W_ra, W);
  return cudaGetLastError();
}

cudaError_t launch_hres_active_grad(const Params& p, const float* dW, float* dW_ra, cudaStream_t st) {
  const size_t n4 = (size_t)p.k * p.k * p.k * p.C / 4;
  const unsigned grid = (unsigned)std::min<size_t>((n4 + 255) / 256, 148 * 16);
  hres_active_grad_kernel<<<grid, 256, 0, st>>>(p, dW, dW_ra);
  return cudaGetLastError();
}

// ============================================================== launchers

cudaError_t launch_wt_prep(const Params& p, const float* W, __nv_bfloat16* Wt, cudaStream_t st) {
  const size_t NC = (size_t)p.N * p.C;
  timing_begin("bwd_wt_prep", st);
  wt_prep_kernel<<<(unsigned)((NC + 63) / 64), 256, 0, st>>>(W, Wt, p.P, NC);
  timing_end(st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const Params& p, const float* W, const float* W_r, __nv_bfloat16* Wt,
                            const float* saved, float* coef, cudaStream_t st) {
  const size_t NC = (size_t)p.N * p.C;
  const size_t T_all = (size_t)p.B * p.S;
  const unsigned nwt = (unsigned)((NC + 63) / 64);
  const unsigned ncoef = (unsigned)((T_all * 16 + 255) / 256);
  timing_begin("bwd_prep", st);
  bwd_prep_kernel<<<nwt + ncoef, 256, 0, st>>>(p, W, W_r, Wt, nwt, saved, coef, T_all);
  timing_end(st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_reduce(const Params& p, const BwdArgs<__nv_bfloat16>& a, bool has_conv, const float* cpart,
                              int conv_rows, int w_ranges, const float* wpart, cudaStream_t st, float* dW_r,
                              const float* cm, float* c_r) {
  const size_t NC = (size_t)p.N * p.C;
  const size_t RNC0 = (size_t)p.P * NC;
  const size_t PNC = RNC0 + (dW_r ? (size_t)p.N * NC : 0);
  timing_begin("bwd_reduce", st);
  if (dW_r) column_sum_kernel<<<p.N, 256, 0, st>>>(cm, (size_t)p.B * p.S, p.N, c_r);
  // conv sums: one thread per output (24 C of them); dW: about two float4 per thread
  const int cblocks = has_conv ? (int)((NTAPS * (size_t)p.C + 255) / 256) : 0;
  const int wblocks = (int)std::min<size_t>(2 * 148 * 8, (PNC / 4 + 511) / 512);
  bwd_reduce_kernel<<<cblocks + std::max(wblocks, 1), 256, 0, st>>>(conv_rows, p.C, cpart, a.dw[0], a.dw[1], a.dw[2],
                                                                   cblocks, w_ranges, PNC, wpart, a.dW, RNC0, NC,
                                                                   dW_r, c_r);
  timing_end(st);
  return cudaGetLastError();
}

}  // namespace xhc
