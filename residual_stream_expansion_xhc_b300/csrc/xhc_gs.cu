// Modified Gram-Schmidt of the TFA components, bf16 state (sm_103a):
//   gs_gram_kernel  per-token Gram matrix of u_0..u_3 (partials per channel block)
//   gs_fold_kernel  per-token Gram-Schmidt coefficients T, H^post' = H^post T
//   gs_bwd_kernel   backward: the Gram term of dL/du through the transposed
//                   convolutions into dout and the conv-weight partials
//
// Method: "xHC: Expanded Hyper-Connections" (qingkeai.online), section
// "Conv / Gram-Schmidt"; section "Temporal Feature Augmentation" for the
// components (causal depthwise convolutions 4, 8, 12, tap tau multiplies
// out[t - tau], zero before the start of each sequence).
#include <algorithm>

#include "xhc_gs.cuh"

namespace xhc {

namespace {

__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// taps of channel c (zero past C): [0,4) K = 4, [4,12) K = 8, [12,24) K = 12
__device__ __forceinline__ void taps_of(const float* const (&w)[3], int c, int C, float (&t)[NTAPS]) {
#pragma unroll
  for (int g = 0; g < NTAPS; ++g) t[g] = 0.0f;
  if (c >= C) return;
#pragma unroll
  for (int q = 0; q < 4; ++q) t[q] = w[0][(size_t)c * 4 + q];
#pragma unroll
  for (int q = 0; q < 8; ++q) t[4 + q] = w[1][(size_t)c * 8 + q];
#pragma unroll
  for (int q = 0; q < 12; ++q) t[12 + q] = w[2][(size_t)c * 12 + q];
}

}  // namespace

// ---------------------------------------------------------------- Gram matrix
//
// CTA = GS_TT tokens of one sequence x GS_CB channels; thread = two adjacent
// channels (fp32x2).  The `out` rows t0 - 11 .. t0 + 31 are staged in shared
// memory; per token the thread forms u_0..u_3 of its channels and the ten
// products, a warp sums them over its 64 channels and the four warps' sums
// are added in a fixed order.

namespace {
constexpr int GG_THREADS = GS_CB / 2;
constexpr int GG_ROWS = GS_TT + HALO;
}  // namespace

__global__ void __launch_bounds__(GG_THREADS) gs_gram_kernel(Params p, const __nv_bfloat16* __restrict__ out,
                                                             const float* __restrict__ w4, const float* __restrict__ w8,
                                                             const float* __restrict__ w12, float* __restrict__ gpart,
                                                             int gcb) {
  __shared__ __align__(16) uint32_t rows[GG_ROWS][GS_CB / 2];   // bf16 pairs
  __shared__ float red[GG_THREADS / 32][GS_TT][10];
  const int S = p.S, C = p.C;
  const int ncs = (S + GS_TT - 1) / GS_TT;
  const int b = blockIdx.x / ncs, t0 = (blockIdx.x % ncs) * GS_TT;
  const int s_end = min(t0 + GS_TT, S);
  const int cb = blockIdx.y, cb0 = cb * GS_CB;
  const size_t seq = (size_t)b * S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < GG_ROWS * (GS_CB / 8); i += GG_THREADS) {
    const int r = i / (GS_CB / 8), q = i % (GS_CB / 8);
    const int t = t0 - HALO + r, c = cb0 + 8 * q;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (t >= 0 && t < S && c < C) v = *reinterpret_cast<const uint4*>(out + (seq + t) * C + c);
    *reinterpret_cast<uint4*>(&rows[r][4 * q]) = v;
  }
  const float* const w[3] = {w4, w8, w12};
  float ta[NTAPS], tb[NTAPS];
  taps_of(w, cb0 + 2 * tid, C, ta);
  taps_of(w, cb0 + 2 * tid + 1, C, tb);
  float2 tp[NTAPS];
#pragma unroll
  for (int g = 0; g < NTAPS; ++g) tp[g] = make_float2(ta[g], tb[g]);
  __syncthreads();
  for (int tt = 0; tt < s_end - t0; ++tt) {
    float2 ow[HALO + 1];
#pragma unroll
    for (int tau = 0; tau <= HALO; ++tau) ow[tau] = bf2_to_f2(rows[tt + HALO - tau][tid]);
    float2 u1 = make_float2(0.0f, 0.0f), u2 = u1, u3 = u1;
#pragma unroll
    for (int tau = 0; tau < 4; ++tau) u1 = __ffma2_rn(tp[tau], ow[tau], u1);
#pragma unroll
    for (int tau = 0; tau < 8; ++tau) u2 = __ffma2_rn(tp[4 + tau], ow[tau], u2);
#pragma unroll
    for (int tau = 0; tau < 12; ++tau) u3 = __ffma2_rn(tp[12 + tau], ow[tau], u3);
    const float2 u[4] = {ow[0], u1, u2, u3};
    float v[10];
    int q = 0;
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = a; c < 4; ++c, ++q) {
        const float2 m = __fmul2_rn(u[a], u[c]);
        v[q] = m.x + m.y;
      }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
      for (int q2 = 0; q2 < 10; ++q2) v[q2] += __shfl_xor_sync(FULL, v[q2], o);
    if (lane == 0)
#pragma unroll
      for (int q2 = 0; q2 < 10; ++q2) red[warp][tt][q2] = v[q2];
  }
  __syncthreads();
  for (int i = tid; i < (s_end - t0) * 10; i += GG_THREADS) {
    const int tt = i / 10, q = i % 10;
    float s = 0.0f;
#pragma unroll
    for (int wq = 0; wq < GG_THREADS / 32; ++wq) s += red[wq][tt][q];
    gpart[((seq + t0 + tt) * gcb + cb) * GS_PSTRIDE + q] = s;
  }
}

int gs_gram_blocks(const Params& p) { return (p.C + GS_CB - 1) / GS_CB; }

cudaError_t launch_gs_gram(const Params& p, const __nv_bfloat16* out, const float* const (&w)[3], float* gpart,
                           cudaStream_t st) {
  const int ncs = (p.S + GS_TT - 1) / GS_TT;
  const dim3 grid((unsigned)(p.B * ncs), (unsigned)gs_gram_blocks(p));
  timing_begin("gs_gram", st);
  gs_gram_kernel<<<grid, GG_THREADS, 0, st>>>(p, out, w[0], w[1], w[2], gpart, gs_gram_blocks(p));
  timing_end(st);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- fold into H^post
//
// One thread per token.

__global__ void __launch_bounds__(256) gs_fold_kernel(Params p, const float* __restrict__ gpart, int gcb,
                                                      float* __restrict__ coef, float* __restrict__ rec, size_t T_all) {
  const size_t tok = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tok >= T_all) return;
  float g[10];
#pragma unroll
  for (int q = 0; q < 10; ++q) g[q] = 0.0f;
  for (int cb = 0; cb < gcb; ++cb) {
    const float* src = gpart + (tok * gcb + cb) * GS_PSTRIDE;
#pragma unroll
    for (int q = 0; q < 10; ++q) g[q] += src[q];
  }
  float M[4][4];
  {
    int q = 0;
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = a; c < 4; ++c, ++q) {
        M[a][c] = g[q];
        M[c][a] = g[q];
      }
  }
  float t[4][4], n[4];
  bool use[4];
  gs_coeffs(M, t, n, use);
  float* hp = coef + tok * COEF_STRIDE + COEF_POST;
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    if (i < p.k) {
      float h[4], o[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) h[c] = hp[4 * i + c];
#pragma unroll
      for (int d = 0; d < 4; ++d) {
        float s = 0.0f;
#pragma unroll
        for (int c = 0; c < 4; ++c) s = fmaf(h[c], t[c][d], s);
        o[d] = s;
      }
#pragma unroll
      for (int d = 0; d < 4; ++d) hp[4 * i + d] = o[d];
    }
  }
  if (rec) {
    float* r = rec + tok * GS_REC;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int d = 0; d < 4; ++d) {
        r[4 * c + d] = t[c][d];
        r[16 + 4 * c + d] = M[c][d];
      }
  }
}

cudaError_t launch_gs_fold(const Params& p, const float* gpart, float* coef, float* rec, cudaStream_t st) {
  const size_t T_all = (size_t)p.B * p.S;
  timing_begin("gs_fold", st);
  gs_fold_kernel<<<(unsigned)((T_all + 255) / 256), 256, 0, st>>>(p, gpart, gs_gram_blocks(p), coef, rec, T_all);
  timing_end(st);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- backward Gram term
//
// CTA = 256 channels (one per thread) x a range of GS_L tokens of one
// sequence, walked downwards from the range's end plus the 11 tokens after it
// that the transposed convolutions reach.  Per token: u_0..u_3 from a window
// of the last 12 `out` values, e = S u, windows of the last e_1..e_3 for the
// transposed convolutions, dout read-modify-write, conv-weight sums in
// registers (one partial row per CTA).

__global__ void __launch_bounds__(256) gs_bwd_kernel(Params p, const __nv_bfloat16* __restrict__ out,
                                                     const float* __restrict__ w4, const float* __restrict__ w8,
                                                     const float* __restrict__ w12, const float* __restrict__ sgram,
                                                     __nv_bfloat16* __restrict__ dout, float* __restrict__ cpart) {
  __shared__ __align__(16) float sg[GS_L + HALO][16];
  const int S = p.S, C = p.C;
  const int nps = (S + GS_L - 1) / GS_L;
  const int b = blockIdx.x / nps, a0 = (blockIdx.x % nps) * GS_L;
  const int bnd = min(a0 + GS_L, S);
  const int top = min(bnd + HALO, S);            // tokens a0 .. top - 1 are walked
  const size_t seq = (size_t)b * S;
  const int c = blockIdx.y * 256 + threadIdx.x;
  const bool ok = c < C;
  for (int i = threadIdx.x; i < (top - a0) * 4; i += 256)
    *reinterpret_cast<float4*>(&sg[i / 4][4 * (i % 4)]) =
        *reinterpret_cast<const float4*>(sgram + (seq + a0 + i / 4) * 16 + 4 * (i % 4));
  const float* const w[3] = {w4, w8, w12};
  float tp[NTAPS];
  taps_of(w, c, C, tp);
  auto out_at = [&](int t) -> float {
    return (ok && t >= 0) ? __bfloat162float(out[(seq + t) * C + c]) : 0.0f;
  };
  float ow[HALO + 1];                             // ow[tau] = out[t - tau]
#pragma unroll
  for (int tau = 0; tau <= HALO; ++tau) ow[tau] = out_at(top - 1 - tau);
  float e1w[4], e2w[8], e3w[12];                  // e_j[t + tau]
#pragma unroll
  for (int q = 0; q < 4; ++q) e1w[q] = 0.0f;
#pragma unroll
  for (int q = 0; q < 8; ++q) e2w[q] = 0.0f;
#pragma unroll
  for (int q = 0; q < 12; ++q) e3w[q] = 0.0f;
  float dw[NTAPS];
#pragma unroll
  for (int g = 0; g < NTAPS; ++g) dw[g] = 0.0f;
  __syncthreads();
  for (int t = top - 1; t >= a0; --t) {
    float u[4];
    u[0] = ow[0];
    u[1] = 0.0f;
    u[2] = 0.0f;
    u[3] = 0.0f;
#pragma unroll
    for (int tau = 0; tau < 4; ++tau) u[1] = fmaf(tp[tau], ow[tau], u[1]);
#pragma unroll
    for (int tau = 0; tau < 8; ++tau) u[2] = fmaf(tp[4 + tau], ow[tau], u[2]);
#pragma unroll
    for (int tau = 0; tau < 12; ++tau) u[3] = fmaf(tp[12 + tau], ow[tau], u[3]);
    const float* s = sg[t - a0];
    float e[4];
#pragma unroll
    for (int d = 0; d < 4; ++d) {
      const float4 r = *reinterpret_cast<const float4*>(s + 4 * d);
      e[d] = fmaf(r.x, u[0], fmaf(r.y, u[1], fmaf(r.z, u[2], r.w * u[3])));
    }
#pragma unroll
    for (int q = 3; q > 0; --q) e1w[q] = e1w[q - 1];
#pragma unroll
    for (int q = 7; q > 0; --q) e2w[q] = e2w[q - 1];
#pragma unroll
    for (int q = 11; q > 0; --q) e3w[q] = e3w[q - 1];
    e1w[0] = e[1];
    e2w[0] = e[2];
    e3w[0] = e[3];
    if (t < bnd && ok) {
      float v = e[0];
#pragma unroll
      for (int tau = 0; tau < 4; ++tau) v = fmaf(tp[tau], e1w[tau], v);
#pragma unroll
      for (int tau = 0; tau < 8; ++tau) v = fmaf(tp[4 + tau], e2w[tau], v);
#pragma unroll
      for (int tau = 0; tau < 12; ++tau) v = fmaf(tp[12 + tau], e3w[tau], v);
      __nv_bfloat16* dst = dout + (seq + t) * C + c;
      *dst = __float2bfloat16_rn(__bfloat162float(*dst) + v);
#pragma unroll
      for (int tau = 0; tau < 4; ++tau) dw[tau] = fmaf(e[1], ow[tau], dw[tau]);
#pragma unroll
      for (int tau = 0; tau < 8; ++tau) dw[4 + tau] = fmaf(e[2], ow[tau], dw[4 + tau]);
#pragma unroll
      for (int tau = 0; tau < 12; ++tau) dw[12 + tau] = fmaf(e[3], ow[tau], dw[12 + tau]);
    }
    // window for t - 1
#pragma unroll
    for (int tau = 0; tau < HALO; ++tau) ow[tau] = ow[tau + 1];
    ow[HALO] = out_at(t - 1 - HALO);
  }
  if (ok) {
    float* row = cpart + (size_t)blockIdx.x * NTAPS * C + c;
#pragma unroll
    for (int g = 0; g < NTAPS; ++g) row[(size_t)g * C] = dw[g];
  }
}

int gs_bwd_rows(const Params& p) { return p.B * ((p.S + GS_L - 1) / GS_L); }

cudaError_t launch_gs_bwd(const Params& p, const __nv_bfloat16* out, const float* const (&w)[3], const float* sgram,
                          __nv_bfloat16* dout, float* cpart, cudaStream_t st) {
  const dim3 grid((unsigned)gs_bwd_rows(p), (unsigned)((p.C + 255) / 256));
  timing_begin("gs_bwd", st);
  gs_bwd_kernel<<<grid, 256, 0, st>>>(p, out, w[0], w[1], w[2], sgram, dout, cpart);
  timing_end(st);
  return cudaGetLastError();
}

}  // namespace xhc
