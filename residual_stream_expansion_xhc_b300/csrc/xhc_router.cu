// Router with per-token active sets, bf16 state (sm_103a):
//   rowsum_kernel          row sums of W_r (the LayerNorm mean term)
//   route_kernel           per token: LayerNorm scores, fixed + top-k slots,
//                          routed write-back scaled into H^post
//   restore_active_kernel  backward of an in-place routed update: the saved
//                          old active rows back into the state at each
//                          token's slots
//
// Method: "xHC: Expanded Hyper-Connections" (qingkeai.online), section "Dense
// read, sparse write": the router reads the LayerNorm-ed whole state and
// scores every stream with a sigmoid; fixed streams are always active, the
// others are chosen per token by top-k; a routed stream's score multiplies
// its new write-back.
//
// The coefficient projection carries W_r as 16 more MMA rows and sums the
// state beside its sum of squares, so it gives, per token, rstd and
// rstd * (W_r v, sum v).  With mean m = sum v / (N C), mean square
// q = 1 / rstd^2 - eps and sd = sqrt(q - m^2 + eps), the scores are
// sigmoid((W_r v - m rs) / sd), rs the row sums of W_r.
#include <algorithm>

#include "xhc_router.cuh"

namespace xhc {

// one block per row; fixed-order tree sum
__global__ void __launch_bounds__(256) rowsum_kernel(const float* __restrict__ W_r, size_t NC, float* __restrict__ rs) {
  __shared__ float part[256];
  const float* row = W_r + (size_t)blockIdx.x * NC;
  float s = 0.0f;
  for (size_t c = threadIdx.x; c < NC; c += 256) s += row[c];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) part[threadIdx.x] += part[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) rs[blockIdx.x] = part[0];
}

struct Fixed {
  int n;
  int s[KMAX];
};

__global__ void __launch_bounds__(64) route_kernel(Params p, const float* __restrict__ zr, const float* __restrict__ rs,
                                                   Fixed fx, int32_t* __restrict__ tok_idx,
                                                   float* __restrict__ rrec, float* __restrict__ coef,
                                                   size_t T_all) {
  const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T_all) return;
  const int N = p.N, k = p.k, P = p.P;
  const float* z = zr + t * (P + 1);
  const float inv = 1.0f / z[P];                               // 1 / rstd
  const float mean = z[N] * inv / (float)((size_t)N * p.C);
  const float msq = inv * inv - p.eps;
  const float sd = sqrtf(fmaxf(msq - mean * mean, 0.0f) + p.eps);
  float s[NMAX], r[NMAX];
#pragma unroll
  for (int n = 0; n < NMAX; ++n) {
    r[n] = n < N ? (z[n] * inv - mean * rs[n]) / sd : 0.0f;
    s[n] = n < N ? sigmoidf_(r[n]) : 0.0f;
  }
  unsigned chosen = 0;
  int slot[KMAX];
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    slot[i] = 0;
    if (i < fx.n) {
      slot[i] = fx.s[i];
      chosen |= 1u << fx.s[i];
    }
  }
  // routed slots: the highest remaining score, the lower index on a tie.
  // The ranking compares the logits r[n]: the sigmoid is monotone, so the
  // order is the scores' order, without the ties that fp32 sigmoid rounding
  // makes of distinct large logits (sigmoid rounds to 1 above about 17).
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    if (i >= fx.n && i < k) {
      int best = -1;
      float bs = 0.0f;
#pragma unroll
      for (int n = 0; n < NMAX; ++n)
        if (n < N && !((chosen >> n) & 1u) && (best < 0 || r[n] > bs)) {
          best = n;
          bs = r[n];
        }
      slot[i] = best;
      chosen |= 1u << best;
    }
  }
  float* rr = rrec + t * (2 * N + 2);
#pragma unroll
  for (int n = 0; n < NMAX; ++n)
    if (n < N) {
      rr[n] = s[n];
      rr[N + n] = r[n];
    }
  rr[2 * N] = mean;
  rr[2 * N + 1] = sd;
  float* hp = coef + t * COEF_STRIDE + COEF_POST;
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    if (i < k) {
      tok_idx[t * k + i] = slot[i];
      if (i >= fx.n) {
        float w = 0.0f;
#pragma unroll
        for (int n = 0; n < NMAX; ++n)
          if (n == slot[i]) w = s[n];
#pragma unroll
        for (int c = 0; c < 4; ++c) hp[4 * i + c] *= w;
      }
    }
  }
}

// Backward: the routed slots' H^post rows scaled by their scores again (the
// coefficient block is rebuilt from the saved logits).
__global__ void __launch_bounds__(64) route_scale_kernel(Params p, const int32_t* __restrict__ tok_idx,
                                                         const float* __restrict__ rrec, int nf,
                                                         float* __restrict__ coef, size_t T_all) {
  const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T_all) return;
  const int k = p.k;
  float* hp = coef + t * COEF_STRIDE + COEF_POST;
  for (int i = nf; i < k; ++i) {
    const float w = rrec[t * (2 * p.N + 2) + tok_idx[t * k + i]];
#pragma unroll
    for (int c = 0; c < 4; ++c) hp[4 * i + c] *= w;
  }
}

cudaError_t launch_route_scale(const Params& p, const int32_t* tok_idx, const float* rrec, int nf, float* coef,
                               cudaStream_t st) {
  const size_t T_all = (size_t)p.B * p.S;
  route_scale_kernel<<<(unsigned)((T_all + 63) / 64), 64, 0, st>>>(p, tok_idx, rrec, nf, coef, T_all);
  return cudaGetLastError();
}

// One thread per 16-byte piece of a saved row: piece q of row (t, i) goes to
// X[t, tok_idx[t, i]].  Slot indices outside [0, N) are skipped.
__global__ void __launch_bounds__(256) restore_active_kernel(uint4* __restrict__ X, const uint4* __restrict__ sa,
                                                             const int32_t* __restrict__ tok_idx, size_t rows,
                                                             int N, int k, int vpr) {
  const size_t n_all = rows * (size_t)vpr;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n_all; e += (size_t)gridDim.x * blockDim.x) {
    const size_t r = e / (size_t)vpr;                  // row t * k + i of saved_active
    const int q = (int)(e - r * (size_t)vpr);
    const int n = __ldg(tok_idx + r);
    if (n < 0 || n >= N) continue;
    const size_t t = r / (size_t)k;
    X[(t * N + n) * vpr + q] = sa[e];
  }
}

cudaError_t launch_restore_active(const Params& p, void* X, const void* saved_active, const int32_t* tok_idx, int sms,
                                  cudaStream_t st) {
  const size_t rows = (size_t)p.B * p.S * p.k;
  const int vpr = p.C * 2 / 16;                        // bf16 rows, C a multiple of 8
  if (rows == 0) return cudaSuccess;
  const size_t n_all = rows * (size_t)vpr;
  const unsigned grid = (unsigned)std::min<size_t>((n_all + 255) / 256, (size_t)sms * 8);
  timing_begin("restore_active", st);
  restore_active_kernel<<<grid, 256, 0, st>>>((uint4*)X, (const uint4*)saved_active, tok_idx, rows, p.N, p.k, vpr);
  timing_end(st);
  return cudaGetLastError();
}

cudaError_t launch_router_rowsums(const Params& p, const float* W_r, float* rs, cudaStream_t st) {
  rowsum_kernel<<<p.N, 256, 0, st>>>(W_r, (size_t)p.N * p.C, rs);
  return cudaGetLastError();
}

cudaError_t launch_route(const Params& p, const float* zr, const float* rs, const int32_t* fixed, int nf,
                         int32_t* tok_idx, float* rrec, float* coef, cudaStream_t st) {
  const size_t T_all = (size_t)p.B * p.S;
  Fixed fx{};
  fx.n = nf;
  for (int i = 0; i < nf && i < KMAX; ++i) fx.s[i] = fixed[i];
  timing_begin("route", st);
  route_kernel<<<(unsigned)((T_all + 63) / 64), 64, 0, st>>>(p, zr, rs, fx, tok_idx, rrec, coef, T_all);
  timing_end(st);
  return cudaGetLastError();
}

}  // namespace xhc
