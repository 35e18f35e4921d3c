// Modified Gram-Schmidt of the four TFA components (optional), bf16 state.
//
// Method: "xHC: Expanded Hyper-Connections" (qingkeai.online), section
// "Conv / Gram-Schmidt": the raw output u_0 is kept and each convolution
// component loses its projections onto the components before it, one at a
// time, so that the write-back combines mutually orthogonal features u~_c.
//
// Per token the orthogonalised components are a fixed combination of the raw
// ones, u~_c = sum_d T[c][d] u_d with T unit lower triangular, and T depends on
// the raw components only through their Gram matrix M[a][b] = <u_a, u_b>
// (sums over the C channels).  The library therefore
//   1. forms M per token (gs_gram_kernel, fp32 sums of fp32 products),
//   2. runs the Gram-Schmidt steps on the coefficient rows (gs_coeffs below):
//      the partly reduced vector v = sum_e r[e] u_e has <v, u~_d> = r M t_d^T
//      and |u~_d|^2 = t_d M t_d^T, so each step of the vector algorithm is
//      taken in the same order on 4-vectors,
//   3. folds T into H^post (H^post' = H^post T), so that the update kernels
//      write sum_d H^post'[i][d] u_d unchanged.
// The backward takes dL/dH^post' (the coefficient dots <G_i, u_d>) back
// through the fold and through the steps (gs_coeffs_reverse) to dL/dM, and
// adds the Gram term dL/du_a += sum_b (dM[a][b] + dM[b][a]) u_b
// (gs_bwd_kernel).
//
// Zero or dependent components: the pages leave them undefined; a projection
// onto u~_d is skipped (coefficient 0) when |u~_d|^2 <= GS_EPS <u_d, u_d>.
#pragma once

#include "xhc_kernels.cuh"

namespace xhc {

constexpr float GS_EPS = 1e-6f;
constexpr int GS_CB = 256;          // channels per CTA of the Gram pass (two per thread)
constexpr int GS_TT = 32;           // tokens per CTA of the Gram pass
constexpr int GS_PSTRIDE = 12;      // floats per (token, channel block) of Gram partials (10 used)
constexpr int GS_REC = 32;          // per-token record: T (16, row-major) then M (16)
constexpr int GS_L = 256;           // tokens per range of the backward Gram term pass

// The Gram-Schmidt steps on coefficient rows.  M: Gram matrix (symmetric).
// t[c]: coefficients of u~_c in the raw components; n[c] = |u~_c|^2;
// use[c]: projections onto u~_c are taken.
__device__ __forceinline__ void gs_coeffs(const float (&M)[4][4], float (&t)[4][4], float (&n)[4], bool (&use)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) t[c][e] = (c == e) ? 1.0f : 0.0f;
  n[0] = M[0][0];
  use[0] = n[0] > GS_EPS * M[0][0];
#pragma unroll
  for (int c = 1; c < 4; ++c) {
    float r[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    r[c] = 1.0f;
#pragma unroll
    for (int d = 0; d < c; ++d) {
      if (use[d]) {
        float q = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float mt = 0.0f;
#pragma unroll
          for (int f = 0; f < 4; ++f) mt = fmaf(M[e][f], t[d][f], mt);
          q = fmaf(r[e], mt, q);
        }
        const float a = q / n[d];
#pragma unroll
        for (int e = 0; e < 4; ++e) r[e] = fmaf(-a, t[d][e], r[e]);
      }
    }
    float nn = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float mr = 0.0f;
#pragma unroll
      for (int f = 0; f < 4; ++f) mr = fmaf(M[e][f], r[f], mr);
      nn = fmaf(r[e], mr, nn);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) t[c][e] = r[e];
    n[c] = nn;
    use[c] = nn > GS_EPS * M[c][c];
  }
}

// Reverse of gs_coeffs: given dL/dt, accumulate dL/dM (dM is overwritten).
// The skip decisions are constants.  For a step r' = r - a t_d with
// a = q / n_d, q = r M t_d^T:
//   da = -<dr', t_d>,  dt_d += -a dr',  dq = da / n_d,  dn_d += -da a / n_d,
//   dr = dr' + dq M t_d^T,  dt_d += dq M r,  dM += dq r t_d^T;
// and n_c = r M r^T gives dr += 2 dn_c M r, dM += dn_c r r^T.
__device__ __forceinline__ void gs_coeffs_reverse(const float (&M)[4][4], const float (&dt_in)[4][4],
                                                  float (&dM)[4][4]) {
  // forward again, keeping each step's row before the step and its a, q
  float t[4][4], n[4];
  bool use[4];
  float rb[4][3][4], av[4][3];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) t[c][e] = (c == e) ? 1.0f : 0.0f;
  n[0] = M[0][0];
  use[0] = n[0] > GS_EPS * M[0][0];
#pragma unroll
  for (int c = 1; c < 4; ++c) {
    float r[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    r[c] = 1.0f;
#pragma unroll
    for (int d = 0; d < c; ++d) {
#pragma unroll
      for (int e = 0; e < 4; ++e) rb[c][d][e] = r[e];
      av[c][d] = 0.0f;
      if (use[d]) {
        float q = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float mt = 0.0f;
#pragma unroll
          for (int f = 0; f < 4; ++f) mt = fmaf(M[e][f], t[d][f], mt);
          q = fmaf(r[e], mt, q);
        }
        const float a = q / n[d];
        av[c][d] = a;
#pragma unroll
        for (int e = 0; e < 4; ++e) r[e] = fmaf(-a, t[d][e], r[e]);
      }
    }
    float nn = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float mr = 0.0f;
#pragma unroll
      for (int f = 0; f < 4; ++f) mr = fmaf(M[e][f], r[f], mr);
      nn = fmaf(r[e], mr, nn);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) t[c][e] = r[e];
    n[c] = nn;
    use[c] = nn > GS_EPS * M[c][c];
  }
  // reverse
  float dt[4][4], dn[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      dt[c][e] = dt_in[c][e];
      dM[c][e] = 0.0f;
    }
#pragma unroll
  for (int c = 3; c >= 1; --c) {
    float dr[4];
    float mr[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float s = 0.0f;
#pragma unroll
      for (int f = 0; f < 4; ++f) s = fmaf(M[e][f], t[c][f], s);
      mr[e] = s;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) dr[e] = fmaf(2.0f * dn[c], mr[e], dt[c][e]);
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
      for (int f = 0; f < 4; ++f) dM[e][f] = fmaf(dn[c] * t[c][e], t[c][f], dM[e][f]);
#pragma unroll
    for (int d = c - 1; d >= 0; --d) {
      if (use[d]) {
        const float a = av[c][d];
        float da = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) da = fmaf(-dr[e], t[d][e], da);
        const float dq = da / n[d];
        dn[d] = fmaf(-da, a / n[d], dn[d]);
        float mt[4], mrb[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float s = 0.0f, u = 0.0f;
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            s = fmaf(M[e][f], t[d][f], s);
            u = fmaf(M[e][f], rb[c][d][f], u);
          }
          mt[e] = s;
          mrb[e] = u;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          dt[d][e] = fmaf(-a, dr[e], dt[d][e]);
          dt[d][e] = fmaf(dq, mrb[e], dt[d][e]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int f = 0; f < 4; ++f) dM[e][f] = fmaf(dq * rb[c][d][e], t[d][f], dM[e][f]);
#pragma unroll
        for (int e = 0; e < 4; ++e) dr[e] = fmaf(dq, mt[e], dr[e]);
      }
    }
  }
  dM[0][0] += dn[0];
}

// Gram partials of every token: gpart[(tok * gcb + cb) * GS_PSTRIDE + q], the
// ten entries M[a][b], a <= b, in the order 00 01 02 03 11 12 13 22 23 33,
// summed over the channels of block cb.
int gs_gram_blocks(const Params& p);
cudaError_t launch_gs_gram(const Params& p, const __nv_bfloat16* out, const float* const (&w)[3], float* gpart,
                           cudaStream_t st);

// Per token: M from the partials, T from M, H^post' = H^post T written over
// the coefficient block's H^post; rec (nullable) [T, GS_REC] gets T and M.
cudaError_t launch_gs_fold(const Params& p, const float* gpart, float* coef, float* rec, cudaStream_t st);

// Backward Gram term: dout[t] += e_0[t] + sum_j sum_tau w_j[tau] e_j[t + tau]
// and dw_j[tau] += sum_t e_j[t] out[t - tau], with e_a = sum_b S[a][b] u_b and
// S = sgram [T, 16] (dM + dM^T).  Conv-weight partials: one row of [24][C] per
// token range, at cpart (rows gs_bwd_rows).
int gs_bwd_rows(const Params& p);
cudaError_t launch_gs_bwd(const Params& p, const __nv_bfloat16* out, const float* const (&w)[3], const float* sgram,
                          __nv_bfloat16* dout, float* cpart, cudaStream_t st);

}  // namespace xhc
