// CUDA-core kernels of the xHC sublayer update (sm_103a).
//
// These kernels serve every shape and both dtypes: they are the fp32 path and
// the fallback for bf16 shapes that the tensor-core kernels do not tile.
// Method: "xHC: Expanded Hyper-Connections" (qingkeai.online), sections
// "Scaling N" (coefficients, Sinkhorn), "Temporal Feature Augmentation"
// (causal depthwise convolutions 4/8/12), "Dense read, sparse write".
#include "xhc_kernels.cuh"

namespace xhc {

// ============================================================== coefficients
//
// One CTA per token: rstd and the P logits z = rstd * (W v) by a block-wide
// reduction over the N*C state entries, then sigmoid / Sinkhorn, then the
// dense read x_in = sum_n hpre[n] X[n] (the token's state is re-read from
// L1/L2, where the first pass left it).

template <typename T>
__global__ void __launch_bounds__(256) coeffs_simt_kernel(Params p, const T* __restrict__ X,
                                                          const float* __restrict__ W,
                                                          float* __restrict__ hpre, float* __restrict__ hpost,
                                                          float* __restrict__ hres, float* __restrict__ saved,
                                                          T* __restrict__ x_in) {
  constexpr int V = Vec<T>::W;
  const size_t t = blockIdx.x;
  const int K = p.N * p.C;
  const T* x = X + t * (size_t)K;
  __shared__ float red[8][PMAX + 1];
  __shared__ float zs[PMAX + 1];
  __shared__ float hpre_s[NMAX];

  float acc[PMAX + 1];
#pragma unroll
  for (int q = 0; q <= PMAX; ++q) acc[q] = 0.0f;
  for (int k0 = threadIdx.x * V; k0 < K; k0 += blockDim.x * V) {
    float xv[V];
    load_vec(x + k0, xv);
#pragma unroll
    for (int e = 0; e < V; ++e) acc[PMAX] = fmaf(xv[e], xv[e], acc[PMAX]);
#pragma unroll
    for (int q = 0; q < PMAX; ++q) {
      if (q < p.P) {
        const float* w = W + (size_t)q * K + k0;
        float wv[V];
#pragma unroll
        for (int e = 0; e < V; e += 4) {
          float4 a = *reinterpret_cast<const float4*>(w + e);
          wv[e] = a.x; wv[e + 1] = a.y; wv[e + 2] = a.z; wv[e + 3] = a.w;
        }
#pragma unroll
        for (int e = 0; e < V; ++e) acc[q] = fmaf(wv[e], xv[e], acc[q]);
      }
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int q = 0; q <= PMAX; ++q) {
    float v = acc[q];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    if (lane == 0) red[warp][q] = v;
  }
  __syncthreads();
  if (threadIdx.x <= PMAX) {
    float s = 0.0f;
    for (int w = 0; w < 8; ++w) s += red[w][threadIdx.x];
    zs[threadIdx.x] = s;
  }
  __syncthreads();
  const float rstd = 1.0f / sqrtf(zs[PMAX] / (float)K + p.eps);
  const int P = p.P, N = p.N, k = p.k;
  if (threadIdx.x < P) {
    const int q = threadIdx.x;
    const float z = rstd * zs[q];
    if (saved) saved[t * (P + 1) + q] = z;
    if (q < N) {
      const float h = sigmoidf_(z);
      hpre_s[q] = h;
      if (hpre) hpre[t * N + q] = h;
    } else if (q < N + 4 * k) {
      if (hpost) hpost[t * 4 * k + (q - N)] = sigmoidf_(z);
    }
  }
  if (threadIdx.x == 0 && saved) saved[t * (P + 1) + P] = rstd;
  if (warp == 0) {
    const int e = lane & 15, i = e >> 2, j = e & 3;
    const bool valid = (i < k) && (j < k);
    const float z = valid ? rstd * zs[N + 4 * k + k * i + j] : 0.0f;
    const float H = sinkhorn16(z, valid, p.iters);
    if (lane < 16 && valid && hres) hres[t * k * k + k * i + j] = H;
  }
  if (x_in == nullptr) return;
  __syncthreads();
  T* xo = x_in + t * (size_t)p.C;
  for (int c0 = threadIdx.x * V; c0 < p.C; c0 += blockDim.x * V) {
    float a[V];
#pragma unroll
    for (int e = 0; e < V; ++e) a[e] = 0.0f;
    for (int n = 0; n < N; ++n) {
      float xv[V];
      load_vec(x + (size_t)n * p.C + c0, xv);
      const float h = hpre_s[n];
#pragma unroll
      for (int e = 0; e < V; ++e) a[e] = fmaf(h, xv[e], a[e]);
    }
    store_vec(xo + c0, a);
  }
}

// ============================================================== sparse update
//
// CTA tile: TT tokens of one sequence x CC = 32 * V channels.  The `out` rows
// of the tile plus an 11-token causal halo and the tile's conv taps are staged
// in shared memory; each warp handles one token at a time, each lane V
// channels.  Coefficients come either from hpost/hres arrays (COEF_ARRAYS) or
// are derived from the saved logits z (sigmoid, Sinkhorn) for the tile.

constexpr int UPD_TT = 32;


template <typename T, bool HAS_CONV>
__global__ void __launch_bounds__(256) update_simt_kernel(Params p, UpdArgs<T> a) {
  constexpr int V = Vec<T>::W;
  constexpr int CC = 32 * V;
  constexpr int CS = PMAX;               // coefficient stride per token
  extern __shared__ float smem[];
  float* out_s = smem;                          // [(TT + HALO) * CC]
  float* w_s = out_s + (UPD_TT + HALO) * CC;    // [NTAPS * CC]
  float* coef_s = w_s + (HAS_CONV ? NTAPS * CC : 0);   // [TT * CS]: hpre | hpost | hres

  const int b = blockIdx.z;
  const int s0 = blockIdx.y * UPD_TT;
  const int c0 = blockIdx.x * CC;
  const int N = p.N, k = p.k, C = p.C, S = p.S;
  const int ntok = min(UPD_TT, S - s0);
  const size_t tok0 = (size_t)b * S + s0;

  // stage out rows [s0 - HALO, s0 + ntok) (zero before the sequence start;
  // absent in the dense-read-only mode)
  for (int r = threadIdx.x / 32; r < UPD_TT + HALO; r += 8) {
    const int s = s0 - HALO + r;
    float v[V];
    if (a.out != nullptr && s >= 0 && s < S && c0 + (threadIdx.x & 31) * V < C) {
      load_vec(a.out + ((size_t)b * S + s) * C + c0 + (threadIdx.x & 31) * V, v);
    } else {
#pragma unroll
      for (int e = 0; e < V; ++e) v[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < V; ++e) out_s[r * CC + (threadIdx.x & 31) * V + e] = v[e];
  }
  if (HAS_CONV) {
    for (int i = threadIdx.x; i < NTAPS * CC; i += blockDim.x) {
      const int g = i / CC, cc = i % CC, c = c0 + cc;
      const int j = g < 4 ? 0 : (g < 12 ? 1 : 2);
      const int K = j == 0 ? 4 : (j == 1 ? 8 : 12);
      const int tau = g - (j == 0 ? 0 : (j == 1 ? 4 : 12));
      w_s[i] = c < C ? a.w[j][(size_t)c * K + tau] : 0.0f;
    }
  }
  // coefficients of the tile's tokens: from the saved logits (sigmoid,
  // Sinkhorn) or from coefficient arrays
  const bool update = a.X_out != nullptr;
  if (a.saved == nullptr) {
    for (int i = threadIdx.x; i < ntok * CS; i += blockDim.x) {
      const int tt = i / CS, q = i % CS;
      float v = 0.0f;
      if (q < N) v = a.hpre ? a.hpre[(tok0 + tt) * N + q] : 0.0f;
      else if (q < N + 4 * k) v = a.hpost ? a.hpost[(tok0 + tt) * 4 * k + (q - N)] : 0.0f;
      else if (q < N + 4 * k + k * k) v = a.hres ? a.hres[(tok0 + tt) * k * k + (q - N - 4 * k)] : 0.0f;
      coef_s[i] = v;
    }
  } else {
    const int P = p.P;
    for (int i = threadIdx.x; i < ntok * CS; i += blockDim.x) {
      const int tt = i / CS, q = i % CS;
      if (q < N + 4 * k) coef_s[i] = sigmoidf_(a.saved[(tok0 + tt) * (P + 1) + q]);
    }
    if (update) {
      // Sinkhorn: two tokens per warp, one per half-warp
      const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
      const int e = lane & 15, i = e >> 2, j = e & 3;
      const bool valid = (i < k) && (j < k);
      for (int tt = warp * 2 + (lane >> 4); tt - (lane >> 4) < ntok; tt += 16) {
        const bool live = tt < ntok;
        const float z = (live && valid) ? a.saved[(tok0 + tt) * (P + 1) + N + 4 * k + k * i + j] : 0.0f;
        const float H = sinkhorn16(z, valid && live, p.iters);
        if (live && valid) coef_s[tt * CS + N + 4 * k + k * i + j] = H;
      }
    }
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cl = lane * V;                       // channel offset inside the tile
  if (c0 + cl >= C) return;
  for (int tt = warp; tt < ntok; tt += 8) {
    const size_t tok = tok0 + tt;
    const float* cf = coef_s + tt * CS;
    const T* xrow = a.X_in + tok * (size_t)N * C + c0 + cl;
    T* yrow = a.X_out + tok * (size_t)N * C + c0 + cl;
    // components
    float u[4][V];
#pragma unroll
    for (int e = 0; e < V; ++e) u[0][e] = out_s[(tt + HALO) * CC + cl + e];
    if (HAS_CONV) {
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int K = j == 0 ? 4 : (j == 1 ? 8 : 12);
        const int g0 = j == 0 ? 0 : (j == 1 ? 4 : 12);
#pragma unroll
        for (int e = 0; e < V; ++e) u[j + 1][e] = 0.0f;
        for (int tau = 0; tau < K; ++tau) {
#pragma unroll
          for (int e = 0; e < V; ++e)
            u[j + 1][e] = fmaf(w_s[(g0 + tau) * CC + cl + e], out_s[(tt + HALO - tau) * CC + cl + e], u[j + 1][e]);
        }
      }
    } else {
#pragma unroll
      for (int j = 1; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < V; ++e) u[j][e] = 0.0f;
    }
    // active rows (before the update)
    float xa[KMAX][V];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) load_vec(xrow + (size_t)p.idx[j] * C, xa[j]);
    }
    if (a.x_in) {
      float acc[V];
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = 0.0f;
      for (int n = 0; n < N; ++n) {
        float xv[V];
        load_vec(xrow + (size_t)n * C, xv);
        const float h = cf[n];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(h, xv[e], acc[e]);
      }
      store_vec(a.x_in + tok * C + c0 + cl, acc);
    }
    if (!update) continue;
    if (a.saved_active) {
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k) store_vec(a.saved_active + (tok * k + j) * C + c0 + cl, xa[j]);
    }
    if (a.copy_inactive) {
      for (int n = 0; n < N; ++n) {
        if (p.is_active[n]) continue;
        float xv[V];
        load_vec(xrow + (size_t)n * C, xv);
        store_vec(yrow + (size_t)n * C, xv);
      }
    }
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      if (i >= k) break;
      float y[V];
      const float* hp = cf + N + 4 * i;
      const float* hr = cf + N + 4 * k + k * i;
#pragma unroll
      for (int e = 0; e < V; ++e) {
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k) acc = fmaf(hr[j], xa[j][e], acc);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc = fmaf(hp[c], u[c][e], acc);
        y[e] = acc;
      }
      store_vec(yrow + (size_t)p.idx[i] * C, y);
    }
  }
}

// ============================================================== TFA components

template <typename T>
__global__ void __launch_bounds__(256) tfa_kernel(Params p, const T* __restrict__ out,
                                                  const float* __restrict__ w4, const float* __restrict__ w8,
                                                  const float* __restrict__ w12, T* __restrict__ u) {
  constexpr int V = Vec<T>::W;
  constexpr int CC = 32 * V;
  extern __shared__ float smem[];
  float* out_s = smem;
  float* w_s = out_s + (UPD_TT + HALO) * CC;
  const int b = blockIdx.z, s0 = blockIdx.y * UPD_TT, c0 = blockIdx.x * CC;
  const int C = p.C, S = p.S;
  const int ntok = min(UPD_TT, S - s0);
  const float* ws[3] = {w4, w8, w12};
  for (int r = threadIdx.x / 32; r < UPD_TT + HALO; r += 8) {
    const int s = s0 - HALO + r;
    float v[V];
    if (s >= 0 && s < S && c0 + (threadIdx.x & 31) * V < C) {
      load_vec(out + ((size_t)b * S + s) * C + c0 + (threadIdx.x & 31) * V, v);
    } else {
#pragma unroll
      for (int e = 0; e < V; ++e) v[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < V; ++e) out_s[r * CC + (threadIdx.x & 31) * V + e] = v[e];
  }
  for (int i = threadIdx.x; i < NTAPS * CC; i += blockDim.x) {
    const int g = i / CC, cc = i % CC, c = c0 + cc;
    const int j = g < 4 ? 0 : (g < 12 ? 1 : 2);
    const int K = j == 0 ? 4 : (j == 1 ? 8 : 12);
    const int tau = g - (j == 0 ? 0 : (j == 1 ? 4 : 12));
    w_s[i] = c < C ? ws[j][(size_t)c * K + tau] : 0.0f;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, cl = lane * V;
  if (c0 + cl >= C) return;
  const size_t plane = (size_t)p.B * S * C;
  for (int tt = warp; tt < ntok; tt += 8) {
    const size_t tok = (size_t)b * S + s0 + tt;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int K = j == 0 ? 4 : (j == 1 ? 8 : 12);
      const int g0 = j == 0 ? 0 : (j == 1 ? 4 : 12);
      float acc[V];
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = 0.0f;
      for (int tau = 0; tau < K; ++tau) {
#pragma unroll
        for (int e = 0; e < V; ++e)
          acc[e] = fmaf(w_s[(g0 + tau) * CC + cl + e], out_s[(tt + HALO - tau) * CC + cl + e], acc[e]);
      }
      store_vec(u + j * plane + tok * C + c0 + cl, acc);
    }
  }
}

// ============================================================== backward, token pass
//
// One CTA per token.  Gradients at the coefficients by reductions over C:
//   dHres[i][j] = <G_i, X[a_j]>, dhpost[i][c] = <G_i, u_c>, dhpre[n] = <dx_in, X[n]>
// (G_i = dX'[a_i]; X is the state before the update), then the reverse pass
// through sigmoid and every Sinkhorn iteration, and dp = rstd * dz,
// alpha = <dz, p> * (-rstd^3 / (N C)).  Record per token (fp32):
//   [ dp (P) | alpha | hpre (N) | hpost (4k) | hres (k^2) ]  -> 2P + 1 floats.

template <typename T, bool HAS_CONV>
__global__ void __launch_bounds__(256) bwd_token_simt_kernel(Params p, BwdArgs<T> a) {
  constexpr int V = Vec<T>::W;
  const size_t t = blockIdx.x;
  const int N = p.N, k = p.k, C = p.C, S = p.S, P = p.P;
  const int s = (int)(t % S);
  const size_t NC = (size_t)N * C;
  __shared__ float red[8][PMAX];
  __shared__ float dsum[PMAX];
  __shared__ float trace[ITERS_MAX][2][32];

  float acc[PMAX];
#pragma unroll
  for (int q = 0; q < PMAX; ++q) acc[q] = 0.0f;
  // accumulator layout: [0, k*k) dHres, [k*k, k*k + 4k) dhpost, then dhpre (N)
  for (int c0 = threadIdx.x * V; c0 < C; c0 += blockDim.x * V) {
    float G[KMAX][V], xa[KMAX][V], u[4][V];
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      if (i < k) {
        load_vec(grad_row(p, a, t, i) + c0, G[i]);
        if (a.saved_active) load_vec(a.saved_active + (t * k + i) * C + c0, xa[i]);
        else load_vec(a.X + t * NC + (size_t)p.idx[i] * C + c0, xa[i]);
      }
    }
    load_vec(a.out + t * C + c0, u[0]);
#pragma unroll
    for (int j = 1; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < V; ++e) u[j][e] = 0.0f;
    if (HAS_CONV) {
      for (int tau = 0; tau < 12 && tau <= s; ++tau) {
        float ov[V];
        load_vec(a.out + (t - tau) * C + c0, ov);
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int K = j == 0 ? 4 : (j == 1 ? 8 : 12);
          if (tau < K) {
#pragma unroll
            for (int e = 0; e < V; ++e) u[j + 1][e] = fmaf(a.w[j][(size_t)(c0 + e) * K + tau], ov[e], u[j + 1][e]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      if (i >= k) break;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j >= k) break;
        float d = 0.0f;
#pragma unroll
        for (int e = 0; e < V; ++e) d = fmaf(G[i][e], xa[j][e], d);
        acc[i * k + j] += d;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float d = 0.0f;
#pragma unroll
        for (int e = 0; e < V; ++e) d = fmaf(G[i][e], u[c][e], d);
        acc[k * k + 4 * i + c] += d;
      }
    }
    if (a.dx_in) {
      float g[V];
      load_vec(a.dx_in + t * C + c0, g);
      for (int n = 0; n < N; ++n) {
        float xv[V];
        const int slot = p.is_active[n];
        if (slot) {
#pragma unroll
          for (int e = 0; e < V; ++e) xv[e] = xa[slot - 1][e];
        } else {
          load_vec(a.X + t * NC + (size_t)n * C + c0, xv);
        }
        float d = 0.0f;
#pragma unroll
        for (int e = 0; e < V; ++e) d = fmaf(g[e], xv[e], d);
#pragma unroll
        for (int q = 0; q < NMAX; ++q)
          if (q == n) acc[k * k + 4 * k + q] += d;
      }
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int q = 0; q < PMAX; ++q) {
    float v = acc[q];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    if (lane == 0) red[warp][q] = v;
  }
  __syncthreads();
  if (threadIdx.x < PMAX) {
    float sum = 0.0f;
    for (int w = 0; w < 8; ++w) sum += red[w][threadIdx.x];
    dsum[threadIdx.x] = sum;
  }
  __syncthreads();
  if (warp != 0) return;
  const float* zt = a.saved + t * (P + 1);
  const float rstd = zt[P];
  float* rec = a.rec + t * (2 * P + 1);
  // H^pre, H^post: dz = dh * h (1 - h)
  float part = 0.0f;       // this lane's share of <dz, p>, p = z / rstd
  for (int q = lane; q < N + 4 * k; q += 32) {
    const float z = zt[q];
    const float h = sigmoidf_(z);
    float dh;
    if (q < N) dh = a.dx_in ? dsum[k * k + 4 * k + q] : 0.0f;
    else dh = dsum[k * k + (q - N)];
    const float dz = dh * h * (1.0f - h);
    rec[q] = rstd * dz;                 // dp
    rec[P + 1 + q] = h;                 // hpre | hpost
    part = fmaf(dz, z / rstd, part);
  }
  // H^res: Sinkhorn forward with the iterates kept, then the reverse pass
  {
    const int e = lane & 15, i = e >> 2, j = e & 3;
    const bool valid = (i < k) && (j < k) && lane < 16;
    const float z = valid ? zt[N + 4 * k + k * i + j] : 0.0f;
    float M0 = sinkhorn_init(z, valid);
    float M = M0;
    for (int it = 0; it < p.iters; ++it)
      M = sinkhorn_step(M, valid, &trace[it][0][lane], &trace[it][1][lane]);
    float g = valid ? dsum[i * k + j] : 0.0f;
    for (int it = p.iters - 1; it >= 0; --it) {
      g = norm_reverse_col(g, trace[it][1][lane], valid);
      g = norm_reverse_row(g, trace[it][0][lane], valid);
    }
    const float dz = g * M0;
    if (valid) {
      const int q = N + 4 * k + k * i + j;
      rec[q] = rstd * dz;
      rec[P + 1 + q] = M;
      part = fmaf(dz, z / rstd, part);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(FULL, part, o);
  if (lane == 0) rec[P] = part * (-(rstd * rstd * rstd) / (float)NC);
}

// ============================================================== backward, dX
//
// dX[n] = sum_q dp[q] W[q][n*C + c] + alpha * X[n] + hpre[n] dx_in
//         + (n inactive ? dX'[n] : sum_i Hres[i][slot(n)] G_i)
// CTA tile: 32 tokens x one stream n x CC = 32 V channels; W's tile columns and
// the tile's token records are staged in shared memory.

template <typename T>
__global__ void __launch_bounds__(256) bwd_dx_simt_kernel(Params p, BwdArgs<T> a) {
  constexpr int V = Vec<T>::W;
  constexpr int CC = 32 * V;
  constexpr int TT = 32;
  extern __shared__ float smem[];
  const int N = p.N, k = p.k, C = p.C, P = p.P;
  const int R = 2 * P + 1;
  float* w_s = smem;                  // [P][CC]
  float* r_s = w_s + PMAX * CC;       // [TT][R]
  const int n = blockIdx.y;
  const int c0 = blockIdx.x * CC;
  const size_t T_all = (size_t)p.B * p.S;
  const size_t t0 = (size_t)blockIdx.z * TT;
  const int ntok = (int)min((size_t)TT, T_all - t0);
  const size_t NC = (size_t)N * C;
  for (int i = threadIdx.x; i < P * CC; i += blockDim.x) {
    const int q = i / CC, cc = i % CC;
    w_s[i] = (c0 + cc < C) ? a.W[(size_t)q * NC + (size_t)n * C + c0 + cc] : 0.0f;
  }
  for (int i = threadIdx.x; i < ntok * R; i += blockDim.x) r_s[i] = a.rec[t0 * R + i];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, cl = lane * V;
  if (c0 + cl >= C) return;
  const int slot = p.is_active[n];
  for (int tt = warp; tt < ntok; tt += 8) {
    const size_t t = t0 + tt;
    const float* r = r_s + tt * R;
    float d[V];
#pragma unroll
    for (int e = 0; e < V; ++e) d[e] = 0.0f;
    for (int q = 0; q < P; ++q) {
      const float g = r[q];
#pragma unroll
      for (int e = 0; e < V; ++e) d[e] = fmaf(g, w_s[q * CC + cl + e], d[e]);
    }
    float xv[V];
    if (slot && a.saved_active) load_vec(a.saved_active + (t * k + (slot - 1)) * C + c0 + cl, xv);
    else load_vec(a.X + t * NC + (size_t)n * C + c0 + cl, xv);
    const float alpha = r[P];
#pragma unroll
    for (int e = 0; e < V; ++e) d[e] = fmaf(alpha, xv[e], d[e]);
    if (a.dx_in) {
      float g[V];
      load_vec(a.dx_in + t * C + c0 + cl, g);
      const float h = r[P + 1 + n];
#pragma unroll
      for (int e = 0; e < V; ++e) d[e] = fmaf(h, g[e], d[e]);
    }
    if (slot) {
      const int j = slot - 1;
      const float* hr = r + P + 1 + N + 4 * k;
      for (int i = 0; i < k; ++i) {
        float g[V];
        load_vec(grad_row(p, a, t, i) + c0 + cl, g);
        const float h = hr[k * i + j];
#pragma unroll
        for (int e = 0; e < V; ++e) d[e] = fmaf(h, g[e], d[e]);
      }
    } else {
      float g[V];
      load_vec(a.dXp + t * NC + (size_t)n * C + c0 + cl, g);
#pragma unroll
      for (int e = 0; e < V; ++e) d[e] += g[e];
    }
    store_vec(a.dX + t * NC + (size_t)n * C + c0 + cl, d);
  }
}

// ============================================================== backward, dW
//
// dW[q][col] = sum over all tokens of dp[t][q] * v[t][col] (v: state before the
// update).  One CTA per 64 columns walks every token in a fixed order: the sum
// is deterministic and needs no partials.

template <typename T>
__global__ void __launch_bounds__(256) bwd_dw_simt_kernel(Params p, BwdArgs<T> a) {
  constexpr int CW = 64, TT = 32;
  __shared__ float v_s[TT][CW];
  __shared__ float g_s[TT][PMAX];
  const int N = p.N, k = p.k, C = p.C, P = p.P, R = 2 * P + 1;
  const size_t NC = (size_t)N * C;
  const size_t col0 = (size_t)blockIdx.x * CW;
  const size_t T_all = (size_t)p.B * p.S;
  const int cw = threadIdx.x % CW;            // column of this thread
  const int qg = threadIdx.x / CW;            // q group: q = qg + 4 m
  float acc[PMAX / 4];
#pragma unroll
  for (int m = 0; m < PMAX / 4; ++m) acc[m] = 0.0f;
  for (size_t t0 = 0; t0 < T_all; t0 += TT) {
    const int ntok = (int)min((size_t)TT, T_all - t0);
    __syncthreads();
    for (int i = threadIdx.x; i < TT * CW; i += blockDim.x) {
      const int tt = i / CW, c = i % CW;
      const size_t col = col0 + c;
      float v = 0.0f;
      if (tt < ntok && col < NC) {
        const size_t t = t0 + tt;
        const int n = (int)(col / C), ch = (int)(col % C);
        const int slot = p.is_active[n];
        if (slot && a.saved_active) v = to_f(a.saved_active[(t * k + (slot - 1)) * C + ch]);
        else v = to_f(a.X[t * NC + col]);
      }
      v_s[tt][c] = v;
    }
    for (int i = threadIdx.x; i < TT * PMAX; i += blockDim.x) {
      const int tt = i / PMAX, q = i % PMAX;
      g_s[tt][q] = (tt < ntok && q < P) ? a.rec[(t0 + tt) * R + q] : 0.0f;
    }
    __syncthreads();
    for (int tt = 0; tt < ntok; ++tt) {
      const float v = v_s[tt][cw];
#pragma unroll
      for (int m = 0; m < PMAX / 4; ++m) acc[m] = fmaf(g_s[tt][qg + 4 * m], v, acc[m]);
    }
  }
  const size_t col = col0 + cw;
  if (col >= NC) return;
#pragma unroll
  for (int m = 0; m < PMAX / 4; ++m) {
    const int q = qg + 4 * m;
    if (q < P) a.dW[(size_t)q * NC + col] = acc[m];
  }
}

// ============================================================== backward, TFA
//
// du_c[t] = sum_i hpost[t][i][c] G_i[t]; dout[t] = du_0[t] + sum_j sum_tau
// w_j[tau] du_j[t + tau] (within the sequence); partial conv-weight gradients
// dw_j[c][tau] = sum_t du_j[t] out[t - tau] per tile of TT tokens, reduced in
// a fixed order afterwards.  CTA tile: TT tokens of one sequence x 32
// channels; thread (channel, token lane).

constexpr int TFA_TT = 128;
constexpr int TFA_CC = 32;

template <typename T, bool HAS_CONV>
__global__ void __launch_bounds__(256) bwd_tfa_simt_kernel(Params p, BwdArgs<T> a, float* __restrict__ partial) {
  extern __shared__ float smem[];
  const int N = p.N, k = p.k, C = p.C, S = p.S, P = p.P, R = 2 * P + 1;
  const int b = blockIdx.z, s0 = blockIdx.y * TFA_TT, c0 = blockIdx.x * TFA_CC;
  const int ntok = min(TFA_TT, S - s0);
  const int nrows = min(TFA_TT + HALO, S - s0);          // du rows needed (forward halo)
  float* du_s = smem;                                     // [TT + HALO][4][CC]
  float* o_s = du_s + (TFA_TT + HALO) * 4 * TFA_CC;       // [TT + HALO][CC]: out rows s0-HALO ..
  float* pw = o_s + (TFA_TT + HALO) * TFA_CC;             // [8 lanes][NTAPS][CC]
  const int cc = threadIdx.x % TFA_CC, lanet = threadIdx.x / TFA_CC;   // 8 token lanes
  const int c = c0 + cc;
  const bool cok = c < C;
  for (int r = lanet; r < TFA_TT + HALO; r += 8) {
    float du[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < nrows && cok) {
      const size_t t = (size_t)b * S + s0 + r;
      const float* hp = a.rec + t * R + P + 1 + N;       // hpost [k][4]
      for (int i = 0; i < k; ++i) {
        const float g = to_f(grad_row(p, a, t, i)[c]);
#pragma unroll
        for (int x = 0; x < 4; ++x) du[x] = fmaf(hp[4 * i + x], g, du[x]);
      }
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) du_s[(r * 4 + x) * TFA_CC + cc] = du[x];
    const int so = s0 - HALO + r;
    o_s[r * TFA_CC + cc] = (so >= 0 && so < S && cok) ? to_f(a.out[((size_t)b * S + so) * C + c]) : 0.0f;
  }
  __syncthreads();
  float pacc[NTAPS];
#pragma unroll
  for (int g = 0; g < NTAPS; ++g) pacc[g] = 0.0f;
  for (int r = lanet; r < ntok; r += 8) {
    float d = du_s[(r * 4 + 0) * TFA_CC + cc];
    if (HAS_CONV) {
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int K = j == 0 ? 4 : (j == 1 ? 8 : 12);
        const int g0 = j == 0 ? 0 : (j == 1 ? 4 : 12);
#pragma unroll
        for (int tau = 0; tau < K; ++tau) {
          if (r + tau < nrows && cok)
            d = fmaf(a.w[j][(size_t)c * K + tau], du_s[((r + tau) * 4 + j + 1) * TFA_CC + cc], d);
          // dw_j[c][tau] += du_j[t] * out[t - tau]
          pacc[g0 + tau] = fmaf(du_s[(r * 4 + j + 1) * TFA_CC + cc], o_s[(r + HALO - tau) * TFA_CC + cc], pacc[g0 + tau]);
        }
      }
    }
    if (cok) from_f(a.dout[((size_t)b * S + s0 + r) * C + c], d);
  }
  if (!HAS_CONV) return;
#pragma unroll
  for (int g = 0; g < NTAPS; ++g) pw[(lanet * NTAPS + g) * TFA_CC + cc] = pacc[g];
  __syncthreads();
  const int tile = blockIdx.z * gridDim.y + blockIdx.y;
  for (int i = threadIdx.x; i < NTAPS * TFA_CC; i += blockDim.x) {
    const int g = i / TFA_CC, ch = i % TFA_CC;
    float sum = 0.0f;
    for (int l = 0; l < 8; ++l) sum += pw[(l * NTAPS + g) * TFA_CC + ch];
    if (c0 + ch < C) partial[((size_t)tile * NTAPS + g) * C + c0 + ch] = sum;
  }
}

// Fixed-order sum of the per-tile conv-weight partials.
__global__ void bwd_tfa_reduce_kernel(int ntiles, int C, const float* __restrict__ partial,
                                      float* __restrict__ dw4, float* __restrict__ dw8, float* __restrict__ dw12) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= NTAPS * C) return;
  const int g = i / C, c = i % C;
  float s = 0.0f;
  for (int tl = 0; tl < ntiles; ++tl) s += partial[((size_t)tl * NTAPS + g) * C + c];
  if (g < 4) dw4[(size_t)c * 4 + g] = s;
  else if (g < 12) dw8[(size_t)c * 8 + (g - 4)] = s;
  else dw12[(size_t)c * 12 + (g - 12)] = s;
}

__global__ void copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = __ldcs(src + i);
}

// ============================================================== launchers

template <typename T>
cudaError_t launch_coeffs_simt(const Params& p, const void* X, const float* W, float* hpre, float* hpost,
                               float* hres, float* saved, void* x_in, cudaStream_t st) {
  const size_t T_all = (size_t)p.B * p.S;
  timing_begin("coeffs_simt", st);
  coeffs_simt_kernel<T><<<(unsigned)T_all, 256, 0, st>>>(p, (const T*)X, W, hpre, hpost, hres, saved, (T*)x_in);
  timing_end(st);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_update_simt(const Params& p, const UpdArgs<T>& a, bool has_conv, cudaStream_t st) {
  constexpr int CC = 32 * Vec<T>::W;
  dim3 grid((p.C + CC - 1) / CC, (p.S + UPD_TT - 1) / UPD_TT, p.B);
  size_t smem = ((UPD_TT + HALO) * CC + (has_conv ? NTAPS * CC : 0) + UPD_TT * PMAX) * sizeof(float);
  timing_begin("update_simt", st);
  if (has_conv) {
    cudaFuncSetAttribute(update_simt_kernel<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    update_simt_kernel<T, true><<<grid, 256, smem, st>>>(p, a);
  } else {
    cudaFuncSetAttribute(update_simt_kernel<T, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    update_simt_kernel<T, false><<<grid, 256, smem, st>>>(p, a);
  }
  timing_end(st);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_tfa(const Params& p, const void* out, const float* w4, const float* w8, const float* w12,
                       void* u, cudaStream_t st) {
  constexpr int CC = 32 * Vec<T>::W;
  dim3 grid((p.C + CC - 1) / CC, (p.S + UPD_TT - 1) / UPD_TT, p.B);
  size_t smem = ((UPD_TT + HALO) * CC + NTAPS * CC) * sizeof(float);
  cudaFuncSetAttribute(tfa_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  timing_begin("tfa", st);
  tfa_kernel<T><<<grid, 256, smem, st>>>(p, (const T*)out, w4, w8, w12, (T*)u);
  timing_end(st);
  return cudaGetLastError();
}

size_t bwd_tfa_partial_floats(const Params& p) {
  const size_t tiles = (size_t)p.B * ((p.S + TFA_TT - 1) / TFA_TT);
  return tiles * NTAPS * (size_t)p.C;
}

template <typename T>
cudaError_t launch_bwd_simt(const Params& p, const BwdArgs<T>& a, bool has_conv, float* partial,
                            bool do_token, cudaStream_t st) {
  const size_t T_all = (size_t)p.B * p.S;
  constexpr int V = Vec<T>::W;
  if (do_token) {
    timing_begin("bwd_token_simt", st);
    if (has_conv) bwd_token_simt_kernel<T, true><<<(unsigned)T_all, 256, 0, st>>>(p, a);
    else bwd_token_simt_kernel<T, false><<<(unsigned)T_all, 256, 0, st>>>(p, a);
    timing_end(st);
  }
  {
    dim3 grid((p.C + TFA_CC - 1) / TFA_CC, (p.S + TFA_TT - 1) / TFA_TT, p.B);
    size_t smem = ((TFA_TT + HALO) * 4 * TFA_CC + (TFA_TT + HALO) * TFA_CC + 8 * NTAPS * TFA_CC) * sizeof(float);
    if (has_conv) {
      cudaFuncSetAttribute(bwd_tfa_simt_kernel<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      timing_begin("bwd_tfa_simt", st);
      bwd_tfa_simt_kernel<T, true><<<grid, 256, smem, st>>>(p, a, partial);
      timing_end(st);
      const int ntiles = (int)(grid.y * grid.z);
      const int n = NTAPS * p.C;
      timing_begin("bwd_tfa_reduce", st);
      bwd_tfa_reduce_kernel<<<(n + 255) / 256, 256, 0, st>>>(ntiles, p.C, partial, a.dw[0], a.dw[1], a.dw[2]);
      timing_end(st);
    } else {
      cudaFuncSetAttribute(bwd_tfa_simt_kernel<T, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      timing_begin("bwd_tfa_simt", st);
      bwd_tfa_simt_kernel<T, false><<<grid, 256, smem, st>>>(p, a, partial);
      timing_end(st);
    }
  }
  {
    const size_t NC = (size_t)p.N * p.C;
    timing_begin("bwd_dw_simt", st);
    bwd_dw_simt_kernel<T><<<(unsigned)((NC + 63) / 64), 256, 0, st>>>(p, a);
    timing_end(st);
  }
  {
    constexpr int CC = 32 * V;
    dim3 grid((p.C + CC - 1) / CC, p.N, (unsigned)((T_all + 31) / 32));
    size_t smem = (PMAX * CC + 32 * (2 * p.P + 1)) * sizeof(float);
    cudaFuncSetAttribute(bwd_dx_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    timing_begin("bwd_dx_simt", st);
    bwd_dx_simt_kernel<T><<<grid, 256, smem, st>>>(p, a);
    timing_end(st);
  }
  return cudaGetLastError();
}

cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, int sms, cudaStream_t st) {
  const size_t n = bytes / 16;
  timing_begin("copy16", st);
  copy16_kernel<<<sms * 4, 512, 0, st>>>((const uint4*)src, (uint4*)dst, n);
  timing_end(st);
  return cudaGetLastError();
}

template cudaError_t launch_coeffs_simt<float>(const Params&, const void*, const float*, float*, float*, float*,
                                               float*, void*, cudaStream_t);
template cudaError_t launch_coeffs_simt<__nv_bfloat16>(const Params&, const void*, const float*, float*, float*,
                                                       float*, float*, void*, cudaStream_t);
template cudaError_t launch_update_simt<float>(const Params&, const UpdArgs<float>&, bool, cudaStream_t);
template cudaError_t launch_update_simt<__nv_bfloat16>(const Params&, const UpdArgs<__nv_bfloat16>&, bool,
                                                       cudaStream_t);
template cudaError_t launch_tfa<float>(const Params&, const void*, const float*, const float*, const float*, void*,
                                       cudaStream_t);
template cudaError_t launch_tfa<__nv_bfloat16>(const Params&, const void*, const float*, const float*,
                                               const float*, void*, cudaStream_t);
template cudaError_t launch_bwd_simt<float>(const Params&, const BwdArgs<float>&, bool, float*, bool, cudaStream_t);
template cudaError_t launch_bwd_simt<__nv_bfloat16>(const Params&, const BwdArgs<__nv_bfloat16>&, bool, float*,
                                                    bool, cudaStream_t);

}  // namespace xhc
