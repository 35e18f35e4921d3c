// Shared device helpers of the xHC update kernels (sm_103a).
//
// Method: "xHC: Expanded Hyper-Connections" (qingkeai.online), sections
// "Scaling N", "Temporal Feature Augmentation", "Dense read, sparse write".
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace xhc {

constexpr int NMAX = 16;             // streams
constexpr int KMAX = 4;              // active streams
constexpr int PMAX = NMAX + 4 * KMAX + KMAX * KMAX;   // 48 logits
constexpr int ITERS_MAX = 64;        // Sinkhorn iterations
constexpr int HALO = 11;             // longest conv (K = 12) reaches 11 tokens back
constexpr int NTAPS = 4 + 8 + 12;    // taps of the three convolutions
constexpr unsigned FULL = 0xffffffffu;

// Kernel-side copy of the problem description.
struct Params {
  int B, S, N, C, k, P, iters;
  float eps;
  int idx[KMAX];
  int is_active[NMAX];    // slot+1 of stream n if active, else 0
  int n_inactive;         // N - k
  int inactive[NMAX];     // the inactive streams in increasing order
};

// ---------------------------------------------------------------- element access

template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int W = 4;     // elements per 16-byte vector
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int W = 8;
};

__device__ __forceinline__ void load_vec(const float* p, float (&v)[4]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void store_vec(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float (&v)[8]) {
  uint4 a = *reinterpret_cast<const uint4*>(p);
  v[0] = bf_lo(a.x); v[1] = bf_hi(a.x); v[2] = bf_lo(a.y); v[3] = bf_hi(a.y);
  v[4] = bf_lo(a.z); v[5] = bf_hi(a.z); v[6] = bf_lo(a.w); v[7] = bf_hi(a.w);
}
__device__ __forceinline__ void store_vec(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 a;
  a.x = pack_bf2(v[0], v[1]); a.y = pack_bf2(v[2], v[3]);
  a.z = pack_bf2(v[4], v[5]); a.w = pack_bf2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = a;
}
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float& d, float x) { d = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16& d, float x) { d = __float2bfloat16_rn(x); }

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

// ---------------------------------------------------------------- Sinkhorn on 16 lanes
//
// One token's k x k H^res is held by a half-warp: lane e = 4 i + j holds entry
// (i, j); entries with i >= k or j >= k are padding and stay 0.  Both halves
// of the warp run the same code (two tokens per warp).  Row sums combine lanes
// differing in bits 0-1, column sums lanes differing in bits 2-3; because IEEE
// addition is commutative every lane of a row (column) obtains the same sum.
// Section "Scaling N": H^res is made doubly stochastic by Sinkhorn
// normalisation; each iteration normalises rows, then columns.

__device__ __forceinline__ float rowsum16(float x) {
  x += __shfl_xor_sync(FULL, x, 1);
  x += __shfl_xor_sync(FULL, x, 2);
  return x;
}
__device__ __forceinline__ float colsum16(float x) {
  x += __shfl_xor_sync(FULL, x, 4);
  x += __shfl_xor_sync(FULL, x, 8);
  return x;
}
__device__ __forceinline__ float max16(float x) {
  x = fmaxf(x, __shfl_xor_sync(FULL, x, 1));
  x = fmaxf(x, __shfl_xor_sync(FULL, x, 2));
  x = fmaxf(x, __shfl_xor_sync(FULL, x, 4));
  x = fmaxf(x, __shfl_xor_sync(FULL, x, 8));
  return x;
}

// M0 = exp(z - max z) over the valid entries.
__device__ __forceinline__ float sinkhorn_init(float z, bool valid) {
  float m = max16(valid ? z : -INFINITY);
  return valid ? expf(z - m) : 0.0f;
}

// One iteration; optionally records the matrices entering each step.
// Each normalisation multiplies by the rounded reciprocal of the sum (one
// reciprocal per row or column instead of a division per entry); the thread
// version below does the same, so both produce identical values.
__device__ __forceinline__ float sinkhorn_step(float M, bool valid, float* before_row, float* before_col) {
  if (before_row) *before_row = M;
  float s = rowsum16(M);
  M = valid ? M * __frcp_rn(s) : 0.0f;
  if (before_col) *before_col = M;
  s = colsum16(M);
  M = valid ? M * __frcp_rn(s) : 0.0f;
  return M;
}

__device__ __forceinline__ float sinkhorn16(float z, bool valid, int iters) {
  float M = sinkhorn_init(z, valid);
  for (int it = 0; it < iters; ++it) M = sinkhorn_step(M, valid, nullptr, nullptr);
  return M;
}

// The same Sinkhorn normalisation with one token's k x k matrix in one
// thread's registers (4 x 4, entries with i >= k or j >= k are padding and
// stay 0).  Sums pair entries as the half-warp version does, ((e0 + e1) +
// (e2 + e3)) along rows and ((r0 + r1) + (r2 + r3)) along columns, so both
// versions produce identical values.  `z` holds the logits row-major (k per
// row, entry (i, j) at z[k i + j]).
__device__ __forceinline__ void sinkhorn_thread(const float* z, int k, int iters, float (&M)[KMAX][KMAX]) {
  float zmax = -INFINITY;
#pragma unroll
  for (int i = 0; i < KMAX; ++i)
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (i < k && j < k) zmax = fmaxf(zmax, z[k * i + j]);
#pragma unroll
  for (int i = 0; i < KMAX; ++i)
#pragma unroll
    for (int j = 0; j < KMAX; ++j) M[i][j] = (i < k && j < k) ? expf(z[k * i + j] - zmax) : 0.0f;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      const float r = __frcp_rn((M[i][0] + M[i][1]) + (M[i][2] + M[i][3]));
#pragma unroll
      for (int j = 0; j < KMAX; ++j) M[i][j] = (i < k && j < k) ? M[i][j] * r : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      const float r = __frcp_rn((M[0][j] + M[1][j]) + (M[2][j] + M[3][j]));
#pragma unroll
      for (int i = 0; i < KMAX; ++i) M[i][j] = (i < k && j < k) ? M[i][j] * r : 0.0f;
    }
  }
}

// Per-token coefficient block written by the coefficient passes and read by
// the update and backward passes: 48 fp32 per token,
//   [ 0, 16) hpre[n]                (n < N, rest 0)
//   [16, 32) hpost[4 i + c]         (i < k, rest 0)
//   [32, 48) Hres[4 i + j]          (i, j < k, rest 0)
constexpr int COEF_STRIDE = 48;
constexpr int COEF_POST = 16;
constexpr int COEF_RES = 32;

// Coefficient block of the tokens of one 256-thread block (a half-warp per
// token: lane e computes hpre[e], hpost[e] and H^res entry e = 4 i + j with the
// shuffle Sinkhorn, which gives the same values as the one-thread version used
// by the forward) from the saved logits [T, P + 1].  `blk` numbers the block
// among those doing this work.
__device__ __forceinline__ void coef_block(const Params& p, const float* __restrict__ saved,
                                           float* __restrict__ coef, size_t T_all, size_t blk) {
  const int lane = threadIdx.x & 31, e = lane & 15;
  const size_t t = (blk * blockDim.x + threadIdx.x) >> 4;
  const bool live = t < T_all;
  const size_t tc = live ? t : 0;
  const int N = p.N, k = p.k, P = p.P;
  const float* z = saved + tc * (P + 1);
  const int i = e >> 2, j = e & 3;
  const bool valid = i < k && j < k;
  const float hpre = e < N ? sigmoidf_(z[e]) : 0.0f;
  const float hpost = e < 4 * k ? sigmoidf_(z[N + e]) : 0.0f;
  const float H = sinkhorn16(valid ? z[N + 4 * k + k * i + j] : 0.0f, valid, p.iters);
  if (!live) return;
  float* cf = coef + t * COEF_STRIDE;
  cf[e] = hpre;
  cf[COEF_POST + e] = hpost;
  cf[COEF_RES + e] = valid ? H : 0.0f;
}

// Reverse of one normalisation y = x / s (s = sum of x along the axis):
// dx = dy / s - sum(dy * x) / s^2 = (dy - sum(dy * x) / s) / s, with 1 / s
// taken once as a rounded reciprocal.
__device__ __forceinline__ float norm_reverse_row(float g, float x, bool valid) {
  const float r = __frcp_rn(rowsum16(x));
  const float gx = rowsum16(g * x);
  return valid ? (g - gx * r) * r : 0.0f;
}
__device__ __forceinline__ float norm_reverse_col(float g, float x, bool valid) {
  const float r = __frcp_rn(colsum16(x));
  const float gx = colsum16(g * x);
  return valid ? (g - gx * r) * r : 0.0f;
}

}  // namespace xhc
