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
  // three tokens per warp-wide transposed sum: 30 of the 32 values
  const int ntok = s_end - t0;
  for (int g0 = 0; g0 < ntok; g0 += 3) {
    float v[32];
    v[30] = 0.0f;
    v[31] = 0.0f;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int tt = g0 + j < ntok ? g0 + j : g0;   // a repeated token past the end is not stored
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
      int q = 0;
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = a; c < 4; ++c, ++q) {
          const float2 m = __fmul2_rn(u[a], u[c]);
          v[10 * j + q] = m.x + m.y;
        }
    }
    // lane l ends with the warp's sum of value l
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < o; ++i) {
        const float send = upper ? v[i] : v[i + o];
        const float keep = upper ? v[i + o] : v[i];
        v[i] = keep + __shfl_xor_sync(FULL, send, o);
      }
    }
    const int tt = g0 + lane / 10;
    if (lane < 30 && tt < ntok) red[warp][tt][lane % 10] = v[0];
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

__global__ void __launch_bounds__(64) gs_fold_kernel(Params p, const float* __restrict__ gpart, int gcb,
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
  // one thread per token, small blocks so that every SM takes part
  gs_fold_kernel<<<(unsigned)((T_all + 63) / 64), 64, 0, st>>>(p, gpart, gs_gram_blocks(p), coef, rec, T_all);
  timing_end(st);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- backward Gram term
//
// CTA = 256 channels (one per thread) x a range of GS_L tokens of one
// sequence, walked downwards from the range's end plus the 11 tokens after it
// that the transposed convolutions reach, in chunks of 32 tokens.  Each
// chunk's `out` rows (with the 11-row halo below), dout rows and S rows are
// brought into shared memory by cp.async one chunk ahead.  Per token: u_0..u_3
// from a window of the last 12 `out` values, e = S u, windows of the last
// e_1..e_3 for the transposed convolutions, dout updated in shared memory and
// written back per chunk with 16-byte stores, conv-weight sums in registers
// (one partial row per CTA).

namespace {
constexpr int GB_TT = 32;
constexpr int GB_ROWS = GB_TT + HALO;
struct GsBwdSmem {
  uint16_t out[2][GB_ROWS][256];
  uint16_t dout[2][GB_TT][256];
  float sg[2][GB_TT][16];
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ float bf_at(const uint16_t v) { return __uint_as_float((uint32_t)v << 16); }
}  // namespace

__global__ void __launch_bounds__(256, 2) gs_bwd_kernel(Params p, const __nv_bfloat16* __restrict__ out,
                                                        const float* __restrict__ w4, const float* __restrict__ w8,
                                                        const float* __restrict__ w12,
                                                        const float* __restrict__ sgram, __nv_bfloat16* __restrict__ dout,
                                                        float* __restrict__ cpart) {
  extern __shared__ __align__(16) uint8_t gb_raw[];
  GsBwdSmem& sm = *reinterpret_cast<GsBwdSmem*>(gb_raw);
  const int S = p.S, C = p.C;
  const int nps = (S + GS_L - 1) / GS_L;
  const int b = blockIdx.x / nps, a0 = (blockIdx.x % nps) * GS_L;
  const int bnd = min(a0 + GS_L, S);
  const int top = min(bnd + HALO, S);            // tokens a0 .. top - 1 are walked
  const int nch = (top - a0 + GB_TT - 1) / GB_TT;
  const size_t seq = (size_t)b * S;
  const int cb0 = blockIdx.y * 256;
  const int tid = threadIdx.x, c = cb0 + tid;
  const bool ok = c < C;
  // chunk j: tokens [lo, hi), hi = top - 32 j
  auto chunk_lo = [&](int j) { return max(top - GB_TT * (j + 1), a0); };
  auto stage = [&](int j) {
    const int hi = top - GB_TT * j, lo = chunk_lo(j), buf = j & 1;
    const int nrows = hi - lo + HALO;
    for (int i = tid; i < nrows * 32; i += 256) {
      const int r = i >> 5, q = i & 31, t = lo - HALO + r, cc = cb0 + 8 * q;
      const bool v = t >= 0 && cc < C;
      cp_async16(&sm.out[buf][r][8 * q], v ? (const void*)(out + (seq + t) * C + cc) : (const void*)out, v);
    }
    const int nd = min(hi, bnd) - lo;
    for (int i = tid; i < nd * 32; i += 256) {
      const int r = i >> 5, q = i & 31, cc = cb0 + 8 * q;
      const bool v = cc < C;
      cp_async16(&sm.dout[buf][r][8 * q], v ? (const void*)(dout + (seq + lo + r) * C + cc) : (const void*)dout, v);
    }
    for (int i = tid; i < (hi - lo) * 4; i += 256)
      cp_async16(&sm.sg[buf][i >> 2][4 * (i & 3)], sgram + (seq + lo + (i >> 2)) * 16 + 4 * (i & 3), true);
    cp_async_commit();
  };
  const float* const w[3] = {w4, w8, w12};
  float tp[NTAPS];
  taps_of(w, c, C, tp);
  float ow[HALO + 1];                             // before token t: ow[tau] = out[t + 1 - tau]
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
  stage(0);
  for (int j = 0; j < nch; ++j) {
    const int hi = top - GB_TT * j, lo = chunk_lo(j), buf = j & 1;
    if (j + 1 < nch) {
      stage(j + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (j == 0) {
      // rows top - 11 .. top - 1 of the first chunk; out[top] is never used
      ow[0] = 0.0f;
#pragma unroll
      for (int tau = 1; tau <= HALO; ++tau) ow[tau] = bf_at(sm.out[0][top - tau - lo + HALO][tid]);
    }
    for (int t = hi - 1; t >= lo; --t) {
#pragma unroll
      for (int tau = 0; tau < HALO; ++tau) ow[tau] = ow[tau + 1];
      ow[HALO] = bf_at(sm.out[buf][t - lo][tid]);   // out[t - 11]
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
      const float* sr = sm.sg[buf][t - lo];
      float e[4];
#pragma unroll
      for (int d = 0; d < 4; ++d) {
        const float4 r = *reinterpret_cast<const float4*>(sr + 4 * d);
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
      if (t < bnd) {
        float v = e[0];
#pragma unroll
        for (int tau = 0; tau < 4; ++tau) v = fmaf(tp[tau], e1w[tau], v);
#pragma unroll
        for (int tau = 0; tau < 8; ++tau) v = fmaf(tp[4 + tau], e2w[tau], v);
#pragma unroll
        for (int tau = 0; tau < 12; ++tau) v = fmaf(tp[12 + tau], e3w[tau], v);
        uint16_t& d = sm.dout[buf][t - lo][tid];
        const __nv_bfloat16 nb = __float2bfloat16_rn(bf_at(d) + v);
        d = *reinterpret_cast<const uint16_t*>(&nb);
#pragma unroll
        for (int tau = 0; tau < 4; ++tau) dw[tau] = fmaf(e[1], ow[tau], dw[tau]);
#pragma unroll
        for (int tau = 0; tau < 8; ++tau) dw[4 + tau] = fmaf(e[2], ow[tau], dw[4 + tau]);
#pragma unroll
        for (int tau = 0; tau < 12; ++tau) dw[12 + tau] = fmaf(e[3], ow[tau], dw[12 + tau]);
      }
    }
    __syncthreads();
    const int nd = min(hi, bnd) - lo;
    for (int i = tid; i < nd * 32; i += 256) {
      const int r = i >> 5, q = i & 31, cc = cb0 + 8 * q;
      if (cc < C)
        *reinterpret_cast<uint4*>(dout + (seq + lo + r) * C + cc) = *reinterpret_cast<const uint4*>(&sm.dout[buf][r][8 * q]);
    }
    __syncthreads();                              // the buffer is staged again two chunks on
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
  const int smem = (int)sizeof(GsBwdSmem);
  cudaFuncSetAttribute(gs_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  timing_begin("gs_bwd", st);
  gs_bwd_kernel<<<grid, 256, smem, st>>>(p, out, w[0], w[1], w[2], sgram, dout, cpart);
  timing_end(st);
  return cudaGetLastError();
}

}  // namespace xhc
