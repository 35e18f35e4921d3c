// Backward of the xHC sublayer update, CUDA-core passes (bf16 state):
//   token pass   per-token gradients at the coefficients, the reverse pass
//                through sigmoid and every Sinkhorn iteration, dp and the
//                rmsnorm term; writes the active-stream mix into dX
//   TFA pass     du_c = sum_i hpost[i][c] G_i, dout (anti-causal transpose of
//                the three convolutions) and conv-weight partial sums
//   reduce       fixed-order sums of the weight-gradient partials
// The tensor-core stream pass (dX for every stream, dW) is in xhc_tc.cu.
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
// operand of dV = dP . W in the stream pass.

__global__ void wt_prep_kernel(const float* __restrict__ W, __nv_bfloat16* __restrict__ Wt, int P, size_t NC) {
  __shared__ float tile[64][65];
  const size_t col0 = (size_t)blockIdx.x * 64;
  for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) {
    const int q = i / 64, c = i % 64;
    tile[q][c] = (q < P && col0 + c < NC) ? W[(size_t)q * NC + col0 + c] : 0.0f;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 32; i += blockDim.x) {
    const int c = i / 32, q2 = (i % 32) * 2;
    if (col0 + c < NC)
      *reinterpret_cast<uint32_t*>(Wt + (col0 + c) * 64 + q2) = pack_bf2(tile[q2][c], tile[q2 + 1][c]);
  }
}

// ============================================================== token pass
//
// One warp per token, lane l owns channels {8 l + 256 m}.  Reads G_i = dX'[a_i],
// the old active rows, `out` (11-token causal window, for u_1..u_3), and with
// dx_in also every stream of X.  Writes, per token:
//   dP[t][0..63]  bf16: dp = rstd * dz (zero padded from P to 64)
//   rec[t]        fp32: [ alpha | hpre (N) | hpost (4k) ], alpha = <dz, p> * (-rstd^3 / (N C))
//   dX[t][a_j]    = sum_i Hres[i][j] G_i      (the mix term of the active streams)

template <bool HAS_CONV>
__global__ void __launch_bounds__(256) bwd_token_kernel(Params p, BwdArgs<__nv_bfloat16> a,
                                                        __nv_bfloat16* __restrict__ dP) {
  constexpr int V = 8;
  extern __shared__ float trace_s[];            // [8 warps][iters][2][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t T_all = (size_t)p.B * p.S;
  const size_t t = (size_t)blockIdx.x * 8 + warp;
  if (t >= T_all) return;                       // the whole warp leaves together
  const int N = p.N, k = p.k, C = p.C, P = p.P, S = p.S;
  const int s = (int)(t % S);
  const size_t NC = (size_t)N * C;
  const float* zt = a.saved + t * (P + 1);
  const float rstd = zt[P];
  float* trace = trace_s + (size_t)warp * p.iters * 64;

  // H^res forward on lanes 0..15 (iterates kept), broadcast to the warp
  const int e = lane & 15, ri = e >> 2, rj = e & 3;
  const bool valid = lane < 16 && ri < k && rj < k;
  const float zres = valid ? zt[N + 4 * k + k * ri + rj] : 0.0f;
  const float M0 = sinkhorn_init(zres, valid);
  float H = M0;
  for (int it = 0; it < p.iters; ++it)
    H = sinkhorn_step(H, valid, &trace[it * 64 + lane], &trace[it * 64 + 32 + lane]);
  float hres[KMAX][KMAX];
#pragma unroll
  for (int i = 0; i < KMAX; ++i)
#pragma unroll
    for (int j = 0; j < KMAX; ++j) hres[i][j] = __shfl_sync(FULL, H, 4 * i + j);

  float d_res[KMAX * KMAX], d_post[4 * KMAX], d_pre[NMAX];
#pragma unroll
  for (int q = 0; q < KMAX * KMAX; ++q) d_res[q] = 0.0f;
#pragma unroll
  for (int q = 0; q < 4 * KMAX; ++q) d_post[q] = 0.0f;
#pragma unroll
  for (int q = 0; q < NMAX; ++q) d_pre[q] = 0.0f;

  for (int c0 = lane * V; c0 < C; c0 += 32 * V) {
    float G[KMAX][V], xa[KMAX][V], u[4][V];
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      if (i < k) {
        load_vec(a.dXp + t * NC + (size_t)p.idx[i] * C + c0, G[i]);
        if (a.saved_active) load_vec(a.saved_active + (t * k + i) * C + c0, xa[i]);
        else load_vec(a.X + t * NC + (size_t)p.idx[i] * C + c0, xa[i]);
      }
    }
    load_vec(a.out + t * C + c0, u[0]);
#pragma unroll
    for (int j = 1; j < 4; ++j)
#pragma unroll
      for (int x = 0; x < V; ++x) u[j][x] = 0.0f;
    if (HAS_CONV) {
      // u_1..u_3 from the causal window out[t - tau], tau < 12, inside the sequence
#pragma unroll
      for (int tau = 0; tau < 12; ++tau) {
        if (tau > s) break;
        float ov[V];
        if (tau == 0) {
#pragma unroll
          for (int x = 0; x < V; ++x) ov[x] = u[0][x];
        } else {
          load_vec(a.out + (t - tau) * C + c0, ov);
        }
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int K = j == 0 ? 4 : (j == 1 ? 8 : 12);
          if (tau < K) {
            const float* w = a.w[j];
#pragma unroll
            for (int x = 0; x < V; ++x) u[j + 1][x] = fmaf(__ldg(w + (size_t)(c0 + x) * K + tau), ov[x], u[j + 1][x]);
          }
        }
      }
    }
    // dots over this lane's channels
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      if (i >= k) break;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j >= k) break;
        float d = 0.0f;
#pragma unroll
        for (int x = 0; x < V; ++x) d = fmaf(G[i][x], xa[j][x], d);
        d_res[i * KMAX + j] += d;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float d = 0.0f;
#pragma unroll
        for (int x = 0; x < V; ++x) d = fmaf(G[i][x], u[c][x], d);
        d_post[4 * i + c] += d;
      }
    }
    if (a.dx_in) {
      float g[V];
      load_vec(a.dx_in + t * C + c0, g);
#pragma unroll
      for (int n = 0; n < NMAX; ++n) {
        if (n >= N) break;
        float xv[V];
        const int slot = p.is_active[n];
        if (slot) {
#pragma unroll
          for (int jj = 0; jj < KMAX; ++jj)
            if (jj == slot - 1)
#pragma unroll
              for (int x = 0; x < V; ++x) xv[x] = xa[jj][x];
        } else {
          load_vec(a.X + t * NC + (size_t)n * C + c0, xv);
        }
        float d = 0.0f;
#pragma unroll
        for (int x = 0; x < V; ++x) d = fmaf(g[x], xv[x], d);
        d_pre[n] += d;
      }
    }
    // mix term of the active streams: dX[a_j] = sum_i Hres[i][j] G_i
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j >= k) break;
      float m[V];
#pragma unroll
      for (int x = 0; x < V; ++x) {
        float acc = 0.0f;
#pragma unroll
        for (int i = 0; i < KMAX; ++i)
          if (i < k) acc = fmaf(hres[i][j], G[i][x], acc);
        m[x] = acc;
      }
      store_vec(a.dX + t * NC + (size_t)p.idx[j] * C + c0, m);
    }
  }
  // warp sums (butterfly: every lane ends with the totals)
#pragma unroll
  for (int q = 0; q < KMAX * KMAX; ++q)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d_res[q] += __shfl_xor_sync(FULL, d_res[q], o);
#pragma unroll
  for (int q = 0; q < 4 * KMAX; ++q)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d_post[q] += __shfl_xor_sync(FULL, d_post[q], o);
  if (a.dx_in) {
#pragma unroll
    for (int q = 0; q < NMAX; ++q)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d_pre[q] += __shfl_xor_sync(FULL, d_pre[q], o);
  }

  // reverse pass through the Sinkhorn iterations (lanes 0..15)
  float gsel = 0.0f;
#pragma unroll
  for (int i = 0; i < KMAX; ++i)
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (4 * i + j == e) gsel = d_res[i * KMAX + j];
  float g = valid ? gsel : 0.0f;
  for (int it = p.iters - 1; it >= 0; --it) {
    g = norm_reverse_col(g, trace[it * 64 + 32 + lane], valid);
    g = norm_reverse_row(g, trace[it * 64 + lane], valid);
  }
  const float dz_res = g * M0;                     // entry (ri, rj) on lane 4 ri + rj

  // logits gradient dz, dp = rstd * dz, <dz, p> with p = z / rstd
  float part = 0.0f;
  float* rec = a.rec + t * (size_t)(1 + N + 4 * k);
  __nv_bfloat16* dprow = dP + t * 64;
  float dpv[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int q = 2 * lane + h;                 // logit handled by this lane
    const int r = q - N - 4 * k;                // H^res entry (r / k, r % k)
    const bool is_res = r >= 0 && q < P;
    const float dzr = __shfl_sync(FULL, dz_res, is_res ? 4 * (r / k) + (r % k) : 0);
    float dz = 0.0f;
    if (q < N) {
      const float hp = sigmoidf_(zt[q]);
      float dh = 0.0f;
#pragma unroll
      for (int n = 0; n < NMAX; ++n)
        if (n == q) dh = d_pre[n];
      dz = a.dx_in ? dh * hp * (1.0f - hp) : 0.0f;
      rec[1 + q] = hp;
    } else if (q < N + 4 * k) {
      const float hq = sigmoidf_(zt[q]);
      float dh = 0.0f;
#pragma unroll
      for (int m = 0; m < 4 * KMAX; ++m)
        if (m == q - N) dh = d_post[m];
      dz = dh * hq * (1.0f - hq);
      rec[1 + q] = hq;
    } else if (is_res) {
      dz = dzr;
    }
    if (q < P) part = fmaf(dz, zt[q] / rstd, part);
    dpv[h] = q < P ? rstd * dz : 0.0f;
  }
  *reinterpret_cast<uint32_t*>(dprow + 2 * lane) = pack_bf2(dpv[0], dpv[1]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(FULL, part, o);
  if (lane == 0) rec[0] = part * (-(rstd * rstd * rstd) / (float)NC);
}

// ============================================================== TFA pass
//
// CTA: one sequence, 64 channels, token blocks of TB = 64 walked in order
// (several per CTA, so that the conv-weight partial sums stay small).
//   phase 1: du_c[t] = sum_i hpost[t][i][c] G_i[t] for t in [s0, s0 + TB + 11)
//            and out[t] for t in [s0 - 11, s0 + TB), staged as fp32
//   phase 2: dout[t] = du_0[t] + sum_j sum_tau w_j[tau] du_j[t + tau]
//            dw_j[tau] += du_j[t] out[t - tau]

constexpr int TFB_TB = 64, TFB_CC = 64, TFB_BLOCKS = 8;

template <bool HAS_CONV>
__global__ void __launch_bounds__(256) bwd_tfa_kernel(Params p, BwdArgs<__nv_bfloat16> a, float* __restrict__ partial) {
  extern __shared__ float sm[];
  constexpr int R = TFB_TB + HALO;
  float* du_s = sm;                          // [4][R][64]
  float* o_s = du_s + 4 * R * TFB_CC;        // [R][64]  rows s0 - 11 ..
  float* red = o_s + R * TFB_CC;             // [4 lanes][24][64]
  const int N = p.N, k = p.k, C = p.C, S = p.S;
  const size_t NC = (size_t)N * C;
  const int b = blockIdx.z, c0 = blockIdx.x * TFB_CC;
  const int rl = 1 + N + 4 * k;
  const int ch = threadIdx.x & 63, tl = threadIdx.x >> 6;      // phase-2 mapping
  float acc[NTAPS];
#pragma unroll
  for (int g = 0; g < NTAPS; ++g) acc[g] = 0.0f;
  float w[NTAPS];
#pragma unroll
  for (int g = 0; g < NTAPS; ++g) {
    const int j = g < 4 ? 0 : (g < 12 ? 1 : 2);
    const int K = j == 0 ? 4 : (j == 1 ? 8 : 12);
    const int tau = g - (j == 0 ? 0 : (j == 1 ? 4 : 12));
    w[g] = HAS_CONV ? __ldg(a.w[j] + (size_t)(c0 + ch) * K + tau) : 0.0f;
  }
  for (int blk = 0; blk < TFB_BLOCKS; ++blk) {
    const int s0 = (blockIdx.y * TFB_BLOCKS + blk) * TFB_TB;
    if (s0 >= S) break;
    __syncthreads();
    // phase 1: 8 threads per row (8 channels each)
    for (int u = threadIdx.x; u < R * 8; u += blockDim.x) {
      const int r = u >> 3, cg = (u & 7) * 8;
      const int st = s0 + r;
      float du[4][8];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int x = 0; x < 8; ++x) du[c][x] = 0.0f;
      if (st < S) {
        const size_t t = (size_t)b * S + st;
        const float* hp = a.rec + t * rl + 1 + N;
        for (int i = 0; i < k; ++i) {
          float gv[8];
          load_vec(a.dXp + t * NC + (size_t)p.idx[i] * C + c0 + cg, gv);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float h = hp[4 * i + c];
#pragma unroll
            for (int x = 0; x < 8; ++x) du[c][x] = fmaf(h, gv[x], du[c][x]);
          }
        }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int x = 0; x < 8; ++x) du_s[(c * R + r) * TFB_CC + cg + x] = du[c][x];
      const int so = s0 - HALO + r;
      float ov[8];
      if (so >= 0 && so < S) {
        load_vec(a.out + ((size_t)b * S + so) * C + c0 + cg, ov);
      } else {
#pragma unroll
        for (int x = 0; x < 8; ++x) ov[x] = 0.0f;
      }
#pragma unroll
      for (int x = 0; x < 8; ++x) o_s[r * TFB_CC + cg + x] = ov[x];
    }
    __syncthreads();
    // phase 2: thread (channel ch, token lane tl)
    for (int r = tl; r < TFB_TB && s0 + r < S; r += 4) {
      float d = du_s[(0 * R + r) * TFB_CC + ch];
      if (HAS_CONV) {
#pragma unroll
        for (int g = 0; g < NTAPS; ++g) {
          const int j = g < 4 ? 0 : (g < 12 ? 1 : 2);
          const int tau = g - (j == 0 ? 0 : (j == 1 ? 4 : 12));
          const float duj_t = du_s[((j + 1) * R + r) * TFB_CC + ch];
          if (s0 + r + tau < S) d = fmaf(w[g], du_s[((j + 1) * R + r + tau) * TFB_CC + ch], d);
          acc[g] = fmaf(duj_t, o_s[(r + HALO - tau) * TFB_CC + ch], acc[g]);
        }
      }
      a.dout[((size_t)b * S + s0 + r) * C + c0 + ch] = __float2bfloat16_rn(d);
    }
  }
  if (!HAS_CONV) return;
  __syncthreads();
#pragma unroll
  for (int g = 0; g < NTAPS; ++g) red[(tl * NTAPS + g) * TFB_CC + ch] = acc[g];
  __syncthreads();
  const int part_row = blockIdx.z * gridDim.y + blockIdx.y;
  for (int u = threadIdx.x; u < NTAPS * TFB_CC; u += blockDim.x) {
    const int g = u / TFB_CC, c = u % TFB_CC;
    const float v = ((red[(0 * NTAPS + g) * TFB_CC + c] + red[(1 * NTAPS + g) * TFB_CC + c]) +
                     red[(2 * NTAPS + g) * TFB_CC + c]) + red[(3 * NTAPS + g) * TFB_CC + c];
    partial[((size_t)part_row * NTAPS + g) * C + c0 + c] = v;
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
      float s = 0.0f;
      for (int r = 0; r < conv_rows; ++r) s += cpart[((size_t)r * NTAPS + g) * C + c];
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

size_t bwd_conv_partial_rows(const Params& p) {
  return (size_t)p.B * ((p.S + TFB_TB * TFB_BLOCKS - 1) / (TFB_TB * TFB_BLOCKS));
}

cudaError_t launch_wt_prep(const Params& p, const float* W, __nv_bfloat16* Wt, cudaStream_t st) {
  const size_t NC = (size_t)p.N * p.C;
  timing_begin("bwd_wt_prep", st);
  wt_prep_kernel<<<(unsigned)((NC + 63) / 64), 256, 0, st>>>(W, Wt, p.P, NC);
  timing_end(st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_token(const Params& p, const BwdArgs<__nv_bfloat16>& a, bool has_conv, __nv_bfloat16* dP,
                             cudaStream_t st) {
  const size_t T_all = (size_t)p.B * p.S;
  const unsigned grid = (unsigned)((T_all + 7) / 8);
  const size_t smem = (size_t)8 * std::max(p.iters, 1) * 64 * sizeof(float);
  timing_begin("bwd_token", st);
  if (has_conv) {
    cudaFuncSetAttribute(bwd_token_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    bwd_token_kernel<true><<<grid, 256, smem, st>>>(p, a, dP);
  } else {
    cudaFuncSetAttribute(bwd_token_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    bwd_token_kernel<false><<<grid, 256, smem, st>>>(p, a, dP);
  }
  timing_end(st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_tfa(const Params& p, const BwdArgs<__nv_bfloat16>& a, bool has_conv, float* cpart,
                           cudaStream_t st) {
  constexpr int R = TFB_TB + HALO;
  const size_t smem = (size_t)(4 * R * TFB_CC + R * TFB_CC + 4 * NTAPS * TFB_CC) * sizeof(float);
  dim3 grid(p.C / TFB_CC, (p.S + TFB_TB * TFB_BLOCKS - 1) / (TFB_TB * TFB_BLOCKS), p.B);
  timing_begin("bwd_tfa", st);
  if (has_conv) {
    cudaFuncSetAttribute(bwd_tfa_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    bwd_tfa_kernel<true><<<grid, 256, smem, st>>>(p, a, cpart);
  } else {
    cudaFuncSetAttribute(bwd_tfa_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    bwd_tfa_kernel<false><<<grid, 256, smem, st>>>(p, a, cpart);
  }
  timing_end(st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_reduce(const Params& p, const BwdArgs<__nv_bfloat16>& a, bool has_conv, const float* cpart,
                              int w_ranges, const float* wpart, cudaStream_t st) {
  const size_t PNC = (size_t)p.P * p.N * p.C;
  timing_begin("bwd_reduce", st);
  bwd_reduce_kernel<<<592, 256, 0, st>>>((int)bwd_conv_partial_rows(p), p.C, has_conv ? cpart : nullptr, a.dw[0],
                                         a.dw[1], a.dw[2], w_ranges, PNC, wpart, a.dW);
  timing_end(st);
  return cudaGetLastError();
}

}  // namespace xhc
