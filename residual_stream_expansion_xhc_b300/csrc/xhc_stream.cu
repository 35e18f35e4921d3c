// Bandwidth-bound CUDA-core passes of the xHC update for bf16 state (sm_103a):
//   coef_kernel       per-token coefficients (sigmoid H^pre / H^post, Sinkhorn
//                     H^res) from saved logits
//   fwd_update_kernel dense read x_in, TFA components and the sparse write
//   bwd_col_kernel    backward: active-stream mix, du = H^post^T G, dout
//                     (transpose of the causal convolutions), conv-weight
//                     partial sums and the per-token coefficient dots
//   bwd_dz_kernel     backward: per-token reverse through sigmoid and every
//                     Sinkhorn iteration; dp and the rmsnorm term
//
// Method: "xHC: Expanded Hyper-Connections" (qingkeai.online research
// retrospective).  Section "Scaling N": the state is N streams of width C;
// H^pre reads the sublayer input from them, H^res (Sinkhorn-normalised) mixes
// them.  Section "Temporal Feature Augmentation": three causal depthwise
// convolutions of kernel size 4, 8, 12 along the sequence, stacked with the
// raw output.  Section "Dense read, sparse write": the input is read from all
// N streams, only the k active streams are rewritten.
//
// Layout of the work.  A CTA owns CB = 256 channels of the state (one channel
// per thread in the channel phases) and walks a contiguous range of chunks of
// TT = 8 tokens (one token per warp in the token phases, eight channels = one
// 16-byte vector per lane).  The causal halo of `out` lives in a ring of rows
// in shared memory, so every row of `out` is read from HBM once per walk.
#include <algorithm>

#include "xhc_debug.cuh"
#include "xhc_gs.cuh"
#include "xhc_stream.cuh"

namespace xhc {

namespace stream {
constexpr int CB = 256;        // channels per CTA
constexpr int TT = 8;          // tokens per chunk
constexpr int THREADS = 256;
constexpr int ORING = 32;      // rows in the `out` ring (power of two)
constexpr int PDOT = 48;       // floats per token and channel block of dots
}  // namespace stream

using namespace stream;

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ void unpack8(const uint4& a, float (&v)[8]) {
  v[0] = bf_lo(a.x); v[1] = bf_hi(a.x); v[2] = bf_lo(a.y); v[3] = bf_hi(a.y);
  v[4] = bf_lo(a.z); v[5] = bf_hi(a.z); v[6] = bf_lo(a.w); v[7] = bf_hi(a.w);
}
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  return make_uint4(pack_bf2(v[0], v[1]), pack_bf2(v[2], v[3]), pack_bf2(v[4], v[5]), pack_bf2(v[6], v[7]));
}
// Global accesses of the big buffers.  In debug builds each is checked
// against the launch's buffer extents (dbg::ok; the caller's source line is
// recorded on a miss) and skipped when it lies outside them.
__device__ __forceinline__ uint4 ld_stream(const __nv_bfloat16* p, int line = __builtin_LINE()) {
  if (!dbg::ok(p, 16, line)) return make_uint4(0, 0, 0, 0);
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream(__nv_bfloat16* p, const uint4& v, int line = __builtin_LINE()) {
  if (!dbg::ok(p, 16, line)) return;
  __stcs(reinterpret_cast<uint4*>(p), v);
}
__device__ __forceinline__ float4 ld_f4(const float* p, int line = __builtin_LINE()) {
  if (!dbg::ok(p, 16, line)) return make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float ld_f(const float* p, int line = __builtin_LINE()) {
  if (!dbg::ok(p, 4, line)) return 0.0f;
  return *p;
}
__device__ __forceinline__ int ld_i(const int32_t* p, int line = __builtin_LINE()) {
  if (!dbg::ok(p, 4, line)) return 0;
  return *p;
}
template <typename V>
__device__ __forceinline__ void st_v(V* p, const V& v, int line = __builtin_LINE()) {
  if (!dbg::ok(p, sizeof(V), line)) return;
  *p = v;
}
__device__ __forceinline__ float bf16_bits(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Conv taps of channel c: w[g], g = 0..3 (K = 4), 4..11 (K = 8), 12..23 (K = 12);
// tap tau multiplies out[t - tau].
__device__ __forceinline__ void load_taps(const float* const (&w)[3], int c, int C, float (&tap)[NTAPS]) {
#pragma unroll
  for (int g = 0; g < NTAPS; ++g) tap[g] = 0.0f;
  if (c >= C) return;
  const float4 a = *reinterpret_cast<const float4*>(w[0] + (size_t)c * 4);
  const float4 b0 = *reinterpret_cast<const float4*>(w[1] + (size_t)c * 8);
  const float4 b1 = *reinterpret_cast<const float4*>(w[1] + (size_t)c * 8 + 4);
  const float4 d0 = *reinterpret_cast<const float4*>(w[2] + (size_t)c * 12);
  const float4 d1 = *reinterpret_cast<const float4*>(w[2] + (size_t)c * 12 + 4);
  const float4 d2 = *reinterpret_cast<const float4*>(w[2] + (size_t)c * 12 + 8);
  const float v[NTAPS] = {a.x,  a.y,  a.z,  a.w,  b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w,
                          d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w, d2.x, d2.y, d2.z, d2.w};
#pragma unroll
  for (int g = 0; g < NTAPS; ++g) tap[g] = v[g];
}

// Ring refill split in two, so that the global load of the row is in flight
// while the warp issues its other loads: warp `warp` fetches row r_beg + warp
// (r_beg + TT rows per chunk, one row per warp) into a register, and commits it
// to the ring later.
__device__ __forceinline__ uint4 fetch_out_row(const __nv_bfloat16* __restrict__ out, size_t seq_base, int S, int C,
                                               int c_lane, int r) {
  uint4 v = make_uint4(0, 0, 0, 0);
  const __nv_bfloat16* q = out + (seq_base + r) * C + c_lane;
  if (r >= 0 && r < S && c_lane < C && dbg::ok(q, 16, __LINE__)) v = *reinterpret_cast<const uint4*>(q);
  return v;
}
__device__ __forceinline__ void commit_out_row(uint16_t (*ring)[CB], int r, int lane, const uint4& v) {
  *reinterpret_cast<uint4*>(&ring[r & (ORING - 1)][8 * lane]) = v;
}

// Rows r_beg .. r_end - 1 (at most 3 TT) of the sequence's `out` into the ring:
// warp w takes rows r_beg + w, r_beg + w + TT, ...; all its loads are issued
// before the first store.  Rows outside [0, S) are zero (the causal padding).
__device__ __forceinline__ void load_out_rows(uint16_t (*ring)[CB], const __nv_bfloat16* __restrict__ out,
                                              size_t seq_base, int S, int C, int c_lane, int r_beg, int r_end,
                                              int warp, int lane) {
  uint4 v[3];
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    const int r = r_beg + warp + q * TT;
    v[q] = r < r_end ? fetch_out_row(out, seq_base, S, C, c_lane, r) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    const int r = r_beg + warp + q * TT;
    if (r < r_end) commit_out_row(ring, r, lane, v[q]);
  }
}

// Work split: the chunks of every sequence, numbered g = b * nch + m (chunk m
// of sequence b), are cut into R contiguous ranges of `per` chunks; CTA
// (r, channel block) walks range r chunk by chunk (the forward upwards, the
// backward downwards), carrying the `out` and du rings from one chunk to the
// next, and restarts only where its range starts or a sequence ends.
struct Walk {
  int nch;        // chunks per sequence
  int ncb;        // channel blocks (grid.y)
  int R;          // ranges = CTAs per channel block (grid.x)
  long per;       // chunks per range
};

Walk make_walk(const Params& p, int sms) {
  Walk w;
  w.nch = (p.S + TT - 1) / TT;
  w.ncb = (p.C + CB - 1) / CB;
  const long total = std::max(1L, (long)p.B * w.nch);
  const long slots = std::max(1L, (long)(2 * sms) / w.ncb);
  const long R = std::min(total, slots);
  w.per = (total + R - 1) / R;
  w.R = (int)((total + w.per - 1) / w.per);   // no empty range
  return w;
}

// ---------------------------------------------------------------- coefficients from saved logits
//
// One thread per token: hpre = sigmoid(z[0:N]), hpost = sigmoid(z[N:N+4k]),
// Hres = Sinkhorn(exp(Z - max Z)) -> coefficient block.

__global__ void __launch_bounds__(256) coef_kernel(Params p, const float* __restrict__ saved, float* __restrict__ coef,
                                                   size_t T_all) {
  coef_block(p, saved, coef, T_all, blockIdx.x);
}

// ---------------------------------------------------------------- forward update
//
// Per chunk: the channel phase computes u_1..u_3 of the chunk (taps and
// `out` from shared memory); the token phase reads the token's N state rows
// once and writes x_in = sum_n hpre[n] X[n], the saved active rows, and
// X'[a_i] = sum_j Hres[i][j] X[a_j] + sum_c hpost[i][c] u_c.

struct FwdSmem {
  uint16_t ring[ORING][CB];          // out rows (bf16 bits)
  float u[3][TT][CB];                // u_1..u_3 of the chunk
  float tap[NTAPS][CB];              // conv taps of the CTA's channels
};

__device__ __forceinline__ void stage_taps(float (*tap_s)[CB], const float* const (&w)[3], int c, int C, int ch) {
  float t[NTAPS];
  load_taps(w, c, C, t);
#pragma unroll
  for (int g = 0; g < NTAPS; ++g) tap_s[g][ch] = t[g];
}

__device__ __forceinline__ float2 fx2(float a) { return make_float2(a, a); }
// bf16 pair (low half first) -> two floats
__device__ __forceinline__ float2 bfx2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// u_1..u_3 of one channel for the chunk tokens t0 .. t0+7 from the ring rows
// t0 - 11 .. t0 + 7 (tokens past the sequence end get values that are never
// read); U is float or bf16 bits.  Tap-outer loops keep eight independent
// accumulators per tap.
template <typename U>
__device__ __forceinline__ void tfa_chunk_s(const uint16_t (*ring)[CB], U (*u_s)[TT][CB], const float (&tap)[NTAPS],
                                            int t0, int ch) {
  float ow[TT + HALO];
#pragma unroll
  for (int i = 0; i < TT + HALO; ++i) ow[i] = bf16_bits(ring[(t0 - HALO + i) & (ORING - 1)][ch]);
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int K = 4 * (j + 1), g0 = (j == 0) ? 0 : (j == 1 ? 4 : 12);
    float u[TT];
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) u[tt] = 0.0f;
#pragma unroll
    for (int tau = 0; tau < K; ++tau)
#pragma unroll
      for (int tt = 0; tt < TT; ++tt) u[tt] = fmaf(tap[g0 + tau], ow[tt + HALO - tau], u[tt]);
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      if constexpr (sizeof(U) == 4) {
        u_s[j][tt][ch] = u[tt];
      } else {
        u_s[j][tt][ch] = __bfloat16_as_ushort(__float2bfloat16_rn(u[tt]));
      }
    }
  }
}

// NI > 0: exactly NI inactive streams, all loaded in one wave; NI = 0: any
// count; NI < 0: per-token active sets (a.tok_idx), the inactive rows by mask.
template <bool HAS_CONV, int NI>
__global__ void __launch_bounds__(THREADS, 2) fwd_update_kernel(Params p, UpdArgs<__nv_bfloat16> a,
                                                                const float* __restrict__ coef, Walk wk) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, ch = threadIdx.x;
  const int N = p.N, k = p.k, C = p.C, S = p.S;
  const int cb0 = blockIdx.y * CB;
  const int c_lane = cb0 + 8 * lane;          // token phases: this lane's 8 channels
  const bool lane_ok = c_lane < C;
  if (HAS_CONV) stage_taps(sm.tap, a.w, cb0 + ch, C, ch);
  const bool need_all = a.x_in != nullptr || a.copy_inactive;
  const long g_beg = (long)blockIdx.x * wk.per;
  const long g_total = (long)p.B * wk.nch;
  const long g_end = g_beg + wk.per < g_total ? g_beg + wk.per : g_total;

  auto channel_phase = [&](int t0) {
    float tap[NTAPS];
#pragma unroll
    for (int g = 0; g < NTAPS; ++g) tap[g] = sm.tap[g][ch];
    tfa_chunk_s<float>(sm.ring, sm.u, tap, t0, ch);
  };

  bool start = true;
  // (b, m) = (g / nch, g mod nch), stepped up with g
  int b = (int)(g_beg / wk.nch), m = (int)(g_beg % wk.nch);
  for (long g = g_beg; g < g_end; ++g, (m + 1 == wk.nch ? (m = 0, ++b) : ++m)) {
    const int t0 = m * TT;
    const int s_end = min(t0 + TT, S);         // tokens of this chunk: t0 .. s_end - 1
    const size_t seq_base = (size_t)b * S;
    const bool has_next = g + 1 < g_end && m + 1 < wk.nch;
    if (start) {
      __syncthreads();                         // the previous walk is done with the ring; taps staged
      if (HAS_CONV) {
        load_out_rows(sm.ring, a.out, seq_base, S, C, c_lane, t0 - HALO, t0 + TT, warp, lane);
        __syncthreads();
        channel_phase(t0);
        __syncthreads();
      }
    }
    start = !has_next;
    {
      const bool refill = HAS_CONV && has_next;
      uint4 next_row;
      if (refill) next_row = fetch_out_row(a.out, seq_base, S, C, c_lane, t0 + TT + warp);
      const int t = t0 + warp;
      if (t < s_end && lane_ok) {
        const size_t tok = seq_base + t;
        const float* cf = coef + tok * COEF_STRIDE;
        const __nv_bfloat16* xrow = a.X_in + tok * (size_t)N * C + c_lane;
        __nv_bfloat16* yrow = a.X_out + tok * (size_t)N * C + c_lane;
        // active streams of this token: the layer's list, or the router's
        // per-token list (NI < 0)
        int ai[KMAX];
        unsigned amask = 0;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          ai[j] = (NI < 0) ? (j < k ? ld_i(a.tok_idx + tok * k + j) : 0) : p.idx[j];
          if (NI < 0 && j < k) amask |= 1u << ai[j];
        }
        uint4 xa[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k) xa[j] = ld_stream(xrow + (size_t)ai[j] * C);
        // x_in partial sums in fp32x2: even and odd inactive rows apart (two
        // independent chains), the active rows into the first
        float2 acc[2][4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          acc[0][x] = make_float2(0.0f, 0.0f);
          acc[1][x] = acc[0][x];
        }
        if (NI < 0 && need_all) {
          // per-token active sets: every stream not in the mask, 8 per wave
#pragma unroll 1
          for (int q0 = 0; q0 < N; q0 += 8) {
            uint4 xr[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (q0 + q < N && !((amask >> (q0 + q)) & 1u)) xr[q] = ld_stream(xrow + (size_t)(q0 + q) * C);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int n = q0 + q;
              if (n < N && !((amask >> n) & 1u)) {
                if (a.x_in) {
                  const float2 h = fx2(ld_f(cf + n));
                  const uint32_t w[4] = {xr[q].x, xr[q].y, xr[q].z, xr[q].w};
#pragma unroll
                  for (int x = 0; x < 4; ++x) acc[q & 1][x] = __ffma2_rn(h, bfx2(w[x]), acc[q & 1][x]);
                }
                if (a.copy_inactive) st_stream(yrow + (size_t)n * C, xr[q]);
              }
            }
          }
        } else if (NI >= 0 && need_all) {
          // the inactive streams, NI (or at most 8) rows per wave of loads
          constexpr int WAVE = NI > 0 ? NI : 8;
          const int ni = NI > 0 ? NI : p.n_inactive;
#pragma unroll 1
          for (int q0 = 0; q0 < ni; q0 += WAVE) {
            uint4 xr[WAVE];
#pragma unroll
            for (int q = 0; q < WAVE; ++q)
              if (q0 + q < ni) xr[q] = ld_stream(xrow + (size_t)p.inactive[q0 + q] * C);
#pragma unroll
            for (int q = 0; q < WAVE; ++q) {
              if (q0 + q < ni) {
                const int n = p.inactive[q0 + q];
                if (a.x_in) {
                  const float2 h = fx2(cf[n]);
                  const uint32_t w[4] = {xr[q].x, xr[q].y, xr[q].z, xr[q].w};
#pragma unroll
                  for (int x = 0; x < 4; ++x) acc[q & 1][x] = __ffma2_rn(h, bfx2(w[x]), acc[q & 1][x]);
                }
                if (a.copy_inactive) st_stream(yrow + (size_t)n * C, xr[q]);
              }
            }
          }
        }
        if (a.x_in) {
#pragma unroll
          for (int j = 0; j < KMAX; ++j) {
            if (j < k) {
              const float2 h = fx2(ld_f(cf + ai[j]));
              const uint32_t w[4] = {xa[j].x, xa[j].y, xa[j].z, xa[j].w};
#pragma unroll
              for (int x = 0; x < 4; ++x) acc[0][x] = __ffma2_rn(h, bfx2(w[x]), acc[0][x]);
            }
          }
          float o[8];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            o[2 * x] = acc[0][x].x + acc[1][x].x;
            o[2 * x + 1] = acc[0][x].y + acc[1][x].y;
          }
          st_stream(a.x_in + tok * C + c_lane, pack8(o));
        }
        if (a.saved_active) {
#pragma unroll
          for (int j = 0; j < KMAX; ++j)
            if (j < k) st_stream(a.saved_active + (tok * k + j) * C + c_lane, xa[j]);
        }
        float u[4][8];
        if (HAS_CONV) {
          unpack8(*reinterpret_cast<const uint4*>(&sm.ring[t & (ORING - 1)][8 * lane]), u[0]);
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            const float4 q0 = *reinterpret_cast<const float4*>(&sm.u[j][warp][8 * lane]);
            const float4 q1 = *reinterpret_cast<const float4*>(&sm.u[j][warp][8 * lane + 4]);
            u[j + 1][0] = q0.x; u[j + 1][1] = q0.y; u[j + 1][2] = q0.z; u[j + 1][3] = q0.w;
            u[j + 1][4] = q1.x; u[j + 1][5] = q1.y; u[j + 1][6] = q1.z; u[j + 1][7] = q1.w;
          }
        } else {
          unpack8(*reinterpret_cast<const uint4*>(a.out + tok * C + c_lane), u[0]);
#pragma unroll
          for (int j = 1; j < 4; ++j)
#pragma unroll
            for (int x = 0; x < 8; ++x) u[j][x] = 0.0f;
        }
        // the k new active rows: independent across i (no early exit), fp32x2
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
          if (i < k) {
            const float4 hp = ld_f4(cf + COEF_POST + 4 * i);
            const float4 hr = ld_f4(cf + COEF_RES + 4 * i);
            const float hrv[4] = {hr.x, hr.y, hr.z, hr.w};
            float2 y[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) y[x] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
              if (j < k) {
                const uint32_t w[4] = {xa[j].x, xa[j].y, xa[j].z, xa[j].w};
#pragma unroll
                for (int x = 0; x < 4; ++x) y[x] = __ffma2_rn(fx2(hrv[j]), bfx2(w[x]), y[x]);
              }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              y[x] = __ffma2_rn(fx2(hp.x), make_float2(u[0][2 * x], u[0][2 * x + 1]), y[x]);
              y[x] = __ffma2_rn(fx2(hp.y), make_float2(u[1][2 * x], u[1][2 * x + 1]), y[x]);
              y[x] = __ffma2_rn(fx2(hp.z), make_float2(u[2][2 * x], u[2][2 * x + 1]), y[x]);
              y[x] = __ffma2_rn(fx2(hp.w), make_float2(u[3][2 * x], u[3][2 * x + 1]), y[x]);
            }
            float o[8];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              o[2 * x] = y[x].x;
              o[2 * x + 1] = y[x].y;
            }
            st_stream(yrow + (size_t)ai[i] * C, pack8(o));
          }
        }
      }
      if (refill) commit_out_row(sm.ring, t0 + TT + warp, lane, next_row);
    }
    if (HAS_CONV) {
      __syncthreads();                         // u of this chunk consumed; next rows in the ring
      if (has_next) channel_phase(t0 + TT);
      __syncthreads();
    }
  }
}

// ---------------------------------------------------------------- backward column pass
//
// CTA = 128 channels, 4 warps, three CTAs per SM; it walks a contiguous range
// of 8-token chunks downwards (the anti-causal direction of the transposed
// convolutions).  Per chunk:
//   token phase (half-warp = token, lane = 8 channels)
//     G_i = dX'[a_i], Xa_j (old active rows) and the token's coefficients,
//           staged in shared memory by cp.async: each warp stages its two
//           token slots of the next chunk as soon as its dots are done, so
//           the loads land while the channel phase runs
//     u_c of the token
//     mix   dX[a_j] = sum_i Hres[i][j] G_i
//     du_c  = sum_i hpost[i][c] G_i: du_1..du_3 -> rings, du_0 kept in registers
//     dots  <G_i, Xa_j>, <G_i, u_c> over the CTA's channels on mma.sync (the
//           rows staged in shared memory) -> pdot[t][channel block]; with
//           dx_in also <dx_in, X_n> (CUDA cores, half-warp sums)
//     dout of the previous chunk's token = du_0 + the convolution parts the
//           channel phase left in shared memory
//     (and the `out` rows the channel phase of this chunk needs next)
//   channel phase (thread = two adjacent channels; threads 0-63 take the K = 4
//   and K = 8 convolutions, threads 64-127 the K = 12 one: 12 taps each, read
//   from a tap-major copy of the conv weights)
//     u_1..u_3 of the next (earlier) chunk
//     convolution parts of dout: sum_tau w_j[tau] du_j[t + tau] (inside the sequence)
//     dw_j[tau] += du_j[t] out[t - tau], in registers for the whole walk
// The du rows of the tokens after a walk's first chunk that its convolutions
// reach (3, 7 and 11 for K = 4, 8, 12) are computed first: the anti-causal
// halo; rows past the sequence end are zeroed.  Conv-weight partials: one row
// per CTA, [R][24][C].

namespace col {
constexpr int CB = 128;                 // channels per CTA
constexpr int THREADS = 128;
constexpr int TT = 8;                   // tokens per chunk (4 warps x 2 half-warps)
constexpr int ORING = 32;
constexpr int D1 = 16, D2 = 16, D3 = 32;   // du ring rows: powers of two >= K_j - 1 + TT
}  // namespace col

// Rows that feed the coefficient dots on the tensor cores are read eight at a
// time by ldmatrix; each such row stores its 16 16-byte chunks rotated by a
// row-specific amount (logical chunk q at physical chunk (q + rot) mod 16), so
// that the eight rows of one ldmatrix fall in eight different bank groups:
//   A rows: G_i of slot s                    rot = i + 4 (s mod 2)
//   B rows: Xa_j (rot j + 1), out (ring, rot 0), u_1..u_3 (rot 5..7)
struct ColSmem {
  uint16_t ring[col::ORING][col::CB];         // out rows (bf16 bits)
  uint32_t u[3][col::TT][col::CB / 2];        // u_1..u_3 of the chunk, bf16 pairs, rotated (they only enter dots)
  float du1[col::D1][col::CB];
  float du2[col::D2][col::CB];
  float du3[col::D3][col::CB];
  float dconv[col::TT][2][col::CB];           // per token slot: convolution parts of dout (K4 + K8 | K12)
  // staged by cp.async one chunk ahead (each warp stages its own two slots
  // once its coefficient dots are done): per token slot
  uint16_t g[col::TT][KMAX][col::CB];         // the G_i rows, rotated (zero where absent)
  uint32_t xa[col::TT][KMAX][col::CB / 2];    // the old active rows Xa_j, rotated
  float cf[col::TT][32];                      // hpost (16) and H^res (16) of the token
};

// ldmatrix of four 8 x 8 bf16 matrices; mma.sync m16n8k16 bf16 -> fp32
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  // rows 8..15 of A are zero
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
               "{%8, %9}, {%0, %1, %2, %3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t rot_chunk(int q, int rot) { return (uint32_t)((q + rot) & 15) << 4; }
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

Walk make_walk_col(const Params& p, int sms) {
  Walk w;
  w.nch = (p.S + col::TT - 1) / col::TT;
  w.ncb = (p.C + col::CB - 1) / col::CB;
  const long total = std::max(1L, (long)p.B * w.nch);
  const long slots = std::max(1L, (long)(3 * sms) / w.ncb);
  const long R = std::min(total, slots);
  w.per = (total + R - 1) / R;
  w.R = (int)((total + w.per - 1) / w.per);
  return w;
}

__device__ __forceinline__ void store8f(float* d, const float2 (&v)[4]) {
  *reinterpret_cast<float4*>(d) = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
  *reinterpret_cast<float4*>(d + 4) = make_float4(v[2].x, v[2].y, v[3].x, v[3].y);
}
__device__ __forceinline__ void unpack8x2(const uint4& a, float2 (&v)[4]) {
  v[0] = make_float2(bf_lo(a.x), bf_hi(a.x));
  v[1] = make_float2(bf_lo(a.y), bf_hi(a.y));
  v[2] = make_float2(bf_lo(a.z), bf_hi(a.z));
  v[3] = make_float2(bf_lo(a.w), bf_hi(a.w));
}
__device__ __forceinline__ uint4 pack8x2(const float2 (&v)[4]) {
  return make_uint4(pack_bf2(v[0].x, v[0].y), pack_bf2(v[1].x, v[1].y), pack_bf2(v[2].x, v[2].y),
                    pack_bf2(v[3].x, v[3].y));
}
// Streaming read that does not allocate in L1.
__device__ __forceinline__ uint4 ld_na(const __nv_bfloat16* p, int line = __builtin_LINE()) {
  uint4 v = make_uint4(0, 0, 0, 0);
  if (!dbg::ok(p, 16, line)) return v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 bf2f(uint32_t w) { return make_float2(bf_lo(w), bf_hi(w)); }
// dot of two 8-vectors held as float2 pairs
__device__ __forceinline__ float dot8(const float2 (&a)[4], const float2 (&b)[4]) {
  float2 s = __fmul2_rn(a[0], b[0]);
  s = __ffma2_rn(a[1], b[1], s);
  s = __ffma2_rn(a[2], b[2], s);
  s = __ffma2_rn(a[3], b[3], s);
  return s.x + s.y;
}
// Sum 16 per-lane values over a half-warp: lane l ends with the sum of value l.
__device__ __forceinline__ float half_transpose_sum16(float (&v)[16], int l16) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool upper = (l16 & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(FULL, send, o);
    }
  }
  return v[0];
}

// ROUTED: per-token active streams a.tok_idx (state before the update in a.X).
template <bool HAS_CONV, bool ROUTED>
__global__ void __launch_bounds__(col::THREADS, 3) bwd_col_kernel(Params p, BwdArgs<__nv_bfloat16> a,
                                                                  const float* __restrict__ coef,
                                                                  float* __restrict__ pdot, float* __restrict__ cpart,
                                                                  const float* __restrict__ taps, Walk wk) {
  constexpr int CBc = col::CB, TTc = col::TT, ORc = col::ORING;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ColSmem& sm = *reinterpret_cast<ColSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int l16 = lane & 15, hw = 2 * warp + (lane >> 4);   // token slot of this half-warp
  const int N = p.N, k = p.k, C = p.C, S = p.S;
  const size_t NC = (size_t)N * C;
  const int cb = blockIdx.y, cb0 = cb * CBc;
  const int c_lane = cb0 + 8 * l16;
  const bool lane_ok = c_lane < C;
  const int pr = threadIdx.x & 63, grp = threadIdx.x >> 6;  // channel phase: pair, convolution group
  const int c2 = cb0 + 2 * pr;
  const bool pair_ok = c2 < C;
  const int ncb = wk.ncb;
  // rows the dots read but no pass writes (channels past C, tokens past the
  // sequence end, the zero row) must hold finite values: start from zero
  for (int q = threadIdx.x; q < (int)(sizeof(ColSmem) / 16); q += col::THREADS)
    reinterpret_cast<uint4*>(smem_raw)[q] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  float2 dw[12];                                            // this group's 12 taps, two channels
#pragma unroll
  for (int q = 0; q < 12; ++q) dw[q] = make_float2(0.0f, 0.0f);
  float2 du0r[4];                                           // du_0 of the token awaiting its dout
#pragma unroll
  for (int q = 0; q < 4; ++q) du0r[q] = make_float2(0.0f, 0.0f);
  bool fin = false;
  size_t fin_tok = 0;

  auto finalize = [&]() {                                   // dout of token fin_tok (slot hw)
    if (fin && lane_ok) {
      const float4 a0 = *reinterpret_cast<const float4*>(&sm.dconv[hw][0][8 * l16]);
      const float4 a1 = *reinterpret_cast<const float4*>(&sm.dconv[hw][0][8 * l16 + 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&sm.dconv[hw][1][8 * l16]);
      const float4 b1 = *reinterpret_cast<const float4*>(&sm.dconv[hw][1][8 * l16 + 4]);
      float2 d[4];
      d[0] = make_float2(du0r[0].x + (a0.x + b0.x), du0r[0].y + (a0.y + b0.y));
      d[1] = make_float2(du0r[1].x + (a0.z + b0.z), du0r[1].y + (a0.w + b0.w));
      d[2] = make_float2(du0r[2].x + (a1.x + b1.x), du0r[2].y + (a1.y + b1.y));
      d[3] = make_float2(du0r[3].x + (a1.z + b1.z), du0r[3].y + (a1.w + b1.w));
      st_stream(a.dout + fin_tok * C + c_lane, pack8x2(d));
    }
    fin = false;
  };

  // du_1..du_3 of a halo token t (lane's channels): rows the convolutions reach
  auto du_halo = [&](size_t seq_base, int t, int s_end) {
    const size_t tok = seq_base + t;
    const float* cf = coef + tok * COEF_STRIDE;
    float2 du[3][4];
#pragma unroll
    for (int c = 0; c < 3; ++c)
#pragma unroll
      for (int q = 0; q < 4; ++q) du[c][q] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      if (i < k) {
        float2 g[4];
        const int ai = ROUTED ? ld_i(a.tok_idx + tok * k + i) : p.idx[i];
        unpack8x2(ld_na(a.dXp + tok * NC + (size_t)ai * C + c_lane), g);
        const float4 hp = ld_f4(cf + COEF_POST + 4 * i);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          du[0][q] = __ffma2_rn(f2(hp.y), g[q], du[0][q]);
          du[1][q] = __ffma2_rn(f2(hp.z), g[q], du[1][q]);
          du[2][q] = __ffma2_rn(f2(hp.w), g[q], du[2][q]);
        }
      }
    }
    const int d = t - s_end;                   // 0 .. 10
    if (d < 3) store8f(&sm.du1[t & (col::D1 - 1)][8 * l16], du[0]);
    if (d < 7) store8f(&sm.du2[t & (col::D2 - 1)][8 * l16], du[1]);
    store8f(&sm.du3[t & (col::D3 - 1)][8 * l16], du[2]);
  };

  // u_1..u_3 of chunk tc from ring rows tc - 11 .. tc + 7 (rows of tokens past
  // the sequence end get finite values that no dot uses: their G rows are zero)
  auto tfa_chunk = [&](const float2 (&tp)[12], int tc) {
    float2 ow[TTc + HALO];
#pragma unroll
    for (int i = 0; i < TTc + HALO; ++i)
      ow[i] = bf2f(*reinterpret_cast<const uint32_t*>(&sm.ring[(tc - HALO + i) & (ORc - 1)][2 * pr]));
    // tap-outer loops: eight independent accumulators per tap
    float2 x[TTc], y[TTc];
#pragma unroll
    for (int tt = 0; tt < TTc; ++tt) {
      x[tt] = make_float2(0.0f, 0.0f);
      y[tt] = x[tt];
    }
    if (grp == 0) {
#pragma unroll
      for (int tau = 0; tau < 4; ++tau)
#pragma unroll
        for (int tt = 0; tt < TTc; ++tt) x[tt] = __ffma2_rn(tp[tau], ow[tt + HALO - tau], x[tt]);
#pragma unroll
      for (int tau = 0; tau < 8; ++tau)
#pragma unroll
        for (int tt = 0; tt < TTc; ++tt) y[tt] = __ffma2_rn(tp[4 + tau], ow[tt + HALO - tau], y[tt]);
#pragma unroll
      for (int tt = 0; tt < TTc; ++tt) {
        sm.u[0][tt][(pr + 20) & 63] = pack_bf2(x[tt].x, x[tt].y);   // rotations 5 and 6
        sm.u[1][tt][(pr + 24) & 63] = pack_bf2(y[tt].x, y[tt].y);
      }
    } else {
#pragma unroll
      for (int tau = 0; tau < 12; ++tau)
#pragma unroll
        for (int tt = 0; tt < TTc; ++tt) x[tt] = __ffma2_rn(tp[tau], ow[tt + HALO - tau], x[tt]);
#pragma unroll
      for (int tt = 0; tt < TTc; ++tt) sm.u[2][tt][(pr + 28) & 63] = pack_bf2(x[tt].x, x[tt].y);   // rotation 7
    }
  };

  // the group's 12 taps of the thread's two channels, from the tap-major
  // copy [24][C] (L1-resident after the first chunk)
  auto load_tap_pairs = [&](float2 (&tp)[12]) {
#pragma unroll
    for (int q = 0; q < 12; ++q) {
      const float* src = taps + (size_t)(12 * grp + q) * C + c2;
      tp[q] = dbg::ok(src, 8, __LINE__) ? __ldg(reinterpret_cast<const float2*>(src)) : make_float2(0.0f, 0.0f);
    }
  };

  // Stage a chunk's per-token rows into the slot buffers by cp.async: the
  // half-warp of slot hw takes token t0s + hw (its lane 8 channels; lanes
  // 0-7 also the token's 32 coefficients).  Rows of absent tokens, channels
  // past C and slots i >= k are zero.  Without convolution branches u_0 (the
  // token's out row) goes to ring row hw.
  auto stage_rows = [&](size_t seq_base_s, int t0s, int s_end_s, const int (&as)[KMAX]) {
    const int ts = t0s + hw;
    const bool ok = ts < s_end_s && lane_ok;
    const size_t tk = seq_base_s + ts;
    const int rot_g = 4 * (hw & 1);
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      uint8_t* gd = reinterpret_cast<uint8_t*>(&sm.g[hw][i][0]) + rot_chunk(l16, i + rot_g);
      uint8_t* xd = reinterpret_cast<uint8_t*>(&sm.xa[hw][i][0]) + rot_chunk(l16, i + 1);
      const __nv_bfloat16* gs = a.dXp + tk * NC + (size_t)as[i] * C + c_lane;
      const __nv_bfloat16* xs = a.saved_active ? a.saved_active + (tk * k + i) * C + c_lane
                                               : a.X + tk * NC + (size_t)as[i] * C + c_lane;
      if (ok && i < k && dbg::ok(gs, 16, __LINE__)) cp_async16(gd, gs);
      else *reinterpret_cast<uint4*>(gd) = make_uint4(0, 0, 0, 0);
      if (ok && i < k && dbg::ok(xs, 16, __LINE__)) cp_async16(xd, xs);
      else *reinterpret_cast<uint4*>(xd) = make_uint4(0, 0, 0, 0);
    }
    if (l16 < 8) {
      const float* cs = coef + tk * COEF_STRIDE + COEF_POST + 4 * l16;
      if (ts < s_end_s && dbg::ok(cs, 16, __LINE__)) cp_async16(&sm.cf[hw][4 * l16], cs);
      else *reinterpret_cast<float4*>(&sm.cf[hw][4 * l16]) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    if (!HAS_CONV) {
      const __nv_bfloat16* os = a.out + tk * C + c_lane;
      if (ok && dbg::ok(os, 16, __LINE__)) cp_async16(&sm.ring[hw][8 * l16], os);
      else *reinterpret_cast<uint4*>(&sm.ring[hw][8 * l16]) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
  };
  bool have_pre = false;                                    // this chunk's rows were staged ahead
  int ai_nx[KMAX];                                          // router: the slots of the next chunk's token
#pragma unroll
  for (int i = 0; i < KMAX; ++i) ai_nx[i] = 0;

  const long g_beg = (long)blockIdx.x * wk.per;
  const long g_total = (long)p.B * wk.nch;
  const long g_end = g_beg + wk.per < g_total ? g_beg + wk.per : g_total;
  bool start = true;
  // (b, m) = (g / nch, g mod nch), stepped down with g
  int b = (int)((g_end - 1) / wk.nch), m = (int)((g_end - 1) % wk.nch);
  for (long g = g_end - 1; g >= g_beg; --g, (m == 0 ? (m = wk.nch - 1, --b) : --m)) {
    const int t0 = m * TTc;
    const int s_end = min(t0 + TTc, S);        // tokens of this chunk: t0 .. s_end - 1
    const size_t seq_base = (size_t)b * S;
    const bool has_next = g - 1 >= g_beg && m > 0;   // the next chunk walked is t0 - TT, same sequence
    if (start) {
      __syncthreads();                         // the previous walk is done with shared memory
      if (HAS_CONV) {
        // out rows t0 - 11 .. t0 + 7 (a half-warp per row), all loads before the stores
        uint4 v[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          const int r = t0 - HALO + hw + 8 * q;
          v[q] = r < t0 + TTc ? fetch_out_row(a.out, seq_base, S, C, c_lane, r) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          const int r = t0 - HALO + hw + 8 * q;
          if (r < t0 + TTc) *reinterpret_cast<uint4*>(&sm.ring[r & (ORc - 1)][8 * l16]) = v[q];
        }
        if (lane_ok) {
          for (int t = s_end + hw; t < min(s_end + HALO, S); t += TTc) du_halo(seq_base, t, s_end);
        }
        // du rows of tokens past the sequence end that this walk's windows
        // reach (t0 + 10, + 14, + 18 for K = 4, 8, 12) are zero: the channel
        // phase then needs no bounds tests.  No later token of the walk is
        // stored in these ring rows while a window still reads them.
        {
          const float2 z[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                               make_float2(0.0f, 0.0f)};
          for (int t = S + hw; t < t0 + TTc + HALO; t += TTc) {
            if (t < t0 + TTc + 3) store8f(&sm.du1[t & (col::D1 - 1)][8 * l16], z);
            if (t < t0 + TTc + 7) store8f(&sm.du2[t & (col::D2 - 1)][8 * l16], z);
            store8f(&sm.du3[t & (col::D3 - 1)][8 * l16], z);
          }
        }
        __syncthreads();
        if (pair_ok) {
          float2 tp[12];
          load_tap_pairs(tp);
          tfa_chunk(tp, t0);
        }
        __syncthreads();
      }
    }
    start = !has_next;
    // ------------------------------------------------ token phase
    const bool refill = HAS_CONV && has_next;
    uint4 next_row;
    if (refill) next_row = fetch_out_row(a.out, seq_base, S, C, c_lane, t0 - TTc - HALO + hw);
    if (HAS_CONV) finalize();                  // dout of the previous chunk's token of this slot
    const int t = t0 + hw;
    const bool tok_ok = t < s_end;             // per half-warp
    const size_t tok = seq_base + (tok_ok ? t : t0);
    int ai[KMAX];                             // this token's active streams
#pragma unroll
    for (int i = 0; i < KMAX; ++i)
      ai[i] = ROUTED ? (have_pre ? ai_nx[i] : (i < k ? ld_i(a.tok_idx + tok * k + i) : 0)) : p.idx[i];
    // this chunk's rows: staged during the previous chunk, or now
    if (!have_pre) stage_rows(seq_base, t0, s_end, ai);
    cp_async_wait_all();
    __syncwarp();
    if (ROUTED && has_next) {
      // the slots of the next chunk's token (a full chunk of this sequence)
      const size_t tn = seq_base + (t0 - TTc) + hw;
#pragma unroll
      for (int i = 0; i < KMAX; ++i) ai_nx[i] = i < k ? ld_i(a.tok_idx + tn * k + i) : 0;
    }
    const float* cs = &sm.cf[hw][0];          // hpost [0, 16), H^res [16, 32)
    float2 G[KMAX][4];
#pragma unroll
    for (int i = 0; i < KMAX; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) G[i][q] = make_float2(0.0f, 0.0f);
    if (tok_ok && lane_ok) {
      const int rot_g = 4 * (hw & 1);
#pragma unroll
      for (int i = 0; i < KMAX; ++i)
        if (i < k)
          unpack8x2(*reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(&sm.g[hw][i][0]) +
                                                    rot_chunk(l16, i + rot_g)),
                    G[i]);
      // active-stream mix: dX[a_j] = sum_i Hres[i][j] G_i
      float hres[KMAX][KMAX];
#pragma unroll
      for (int i = 0; i < KMAX; ++i) {
        const float4 h = *reinterpret_cast<const float4*>(cs + 16 + 4 * i);
        hres[i][0] = h.x; hres[i][1] = h.y; hres[i][2] = h.z; hres[i][3] = h.w;
      }
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
          float2 mx[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) mx[q] = __fmul2_rn(f2(hres[0][j]), G[0][q]);   // k >= 1
#pragma unroll
          for (int i = 1; i < KMAX; ++i)
            if (i < k)
#pragma unroll
              for (int q = 0; q < 4; ++q) mx[q] = __ffma2_rn(f2(hres[i][j]), G[i][q], mx[q]);
          st_stream(a.dX + tok * NC + (size_t)ai[j] * C + c_lane, pack8x2(mx));
        }
      }
      // du_c = sum_i hpost[i][c] G_i
      float2 du[4][4];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int q = 0; q < 4; ++q) du[c][q] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int i = 0; i < KMAX; ++i) {
        if (i < k) {
          const float4 hp = *reinterpret_cast<const float4*>(cs + 4 * i);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            du[0][q] = __ffma2_rn(f2(hp.x), G[i][q], du[0][q]);
            du[1][q] = __ffma2_rn(f2(hp.y), G[i][q], du[1][q]);
            du[2][q] = __ffma2_rn(f2(hp.z), G[i][q], du[2][q]);
            du[3][q] = __ffma2_rn(f2(hp.w), G[i][q], du[3][q]);
          }
        }
      }
      if (HAS_CONV) {
#pragma unroll
        for (int q = 0; q < 4; ++q) du0r[q] = du[0][q];
        store8f(&sm.du1[t & (col::D1 - 1)][8 * l16], du[1]);
        store8f(&sm.du2[t & (col::D2 - 1)][8 * l16], du[2]);
        store8f(&sm.du3[t & (col::D3 - 1)][8 * l16], du[3]);
      } else {
        st_stream(a.dout + tok * C + c_lane, pack8x2(du[0]));
      }
    }
    if (HAS_CONV && tok_ok) {
      fin = true;
      fin_tok = tok;
    }
    // Coefficient dots of this CTA's channels, per token: [0,16) <G_i, Xa_j>
    // at 4i+j, [16,32) <G_i, u_c> at 16+4i+c.  Per warp (two tokens, slots
    // 2w and 2w+1) they are two small contractions over the 128 channels,
    //   D_T[i][n] = sum_ch G_T,i[ch] Y_T,n[ch],  Y_T = (Xa_0..Xa_3, u_0..u_3),
    // run as mma.sync m16n8k16 (bf16 in, fp32 sums): A rows 0-3 hold G of
    // slot 2w, rows 4-7 G of slot 2w+1 (rows 8-15 zero), B holds one token's
    // Y; the token's own rows of D are kept.  The bf16 products are exact and
    // the sums are fp32, as with the CUDA-core dots they replace.
    {
      // the staged rows (without convolution branches u_0 = the token's out
      // row, staged in the unused ring; ring[ORING - 1] stays zero)
      const int mq = lane >> 3, rr = lane & 7;  // ldmatrix: this lane addresses row rr of matrix mq
      const int sa = 2 * warp + (rr >> 2), ia = rr & 3;
      const uint32_t a_row = smem_u32(&sm.g[sa][ia][0]);
      const int a_rot = mq + ia + 4 * (sa & 1);
      uint32_t b_row[2];
      int b_rot;
#pragma unroll
      for (int T = 0; T < 2; ++T) {
        const int sb = 2 * warp + T;
        if (rr < 4) {
          b_row[T] = smem_u32(&sm.xa[sb][rr][0]);
        } else if (rr == 4) {
          b_row[T] = HAS_CONV ? smem_u32(&sm.ring[(t0 + sb) & (ORc - 1)][0]) : smem_u32(&sm.ring[sb][0]);
        } else {
          b_row[T] = HAS_CONV ? smem_u32(&sm.u[rr - 5][sb][0]) : smem_u32(&sm.ring[ORc - 1][0]);
        }
      }
      b_rot = mq + (rr < 4 ? rr + 1 : (rr == 4 ? 0 : (HAS_CONV ? rr : 0)));
      float dA[4] = {0.0f, 0.0f, 0.0f, 0.0f}, dB[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int pp = 0; pp < CBc / 32; ++pp) {   // two 16-channel K steps per ldmatrix
        uint32_t fa[4], fb[4];
        ldsm_x4(a_row + rot_chunk(4 * pp, a_rot), fa);
        ldsm_x4(b_row[0] + rot_chunk(4 * pp, b_rot), fb);
        mma_16816(dA, fa[0], fa[1], fb[0], fb[1]);
        mma_16816(dA, fa[2], fa[3], fb[2], fb[3]);
        ldsm_x4(b_row[1] + rot_chunk(4 * pp, b_rot), fb);
        mma_16816(dB, fa[0], fa[1], fb[0], fb[1]);
        mma_16816(dB, fa[2], fa[3], fb[2], fb[3]);
      }
      // lane = 4 g + t holds D[g][2t], D[g][2t + 1]; rows g = 0-3 are slot 2w's
      // tokens (from dA), rows 4-7 slot 2w+1's (from dB): i = g mod 4
      const float2 r = lane < 16 ? make_float2(dA[0], dA[1]) : make_float2(dB[0], dB[1]);
      const int gi = (lane >> 2) & 3, n0 = 2 * (lane & 3);
      const int at = n0 < 4 ? 4 * gi + n0 : 16 + 4 * gi + (n0 - 4);
      if (tok_ok) st_v(reinterpret_cast<float2*>(pdot + (tok * ncb + cb) * PDOT + at), r);
    }
    // the warp's slots are read: stage the next chunk of the walk into them,
    // to land while the channel phase runs
    __syncwarp();
    have_pre = has_next;
    if (has_next) {
      int an[KMAX];
#pragma unroll
      for (int i = 0; i < KMAX; ++i) an[i] = ROUTED ? ai_nx[i] : p.idx[i];
      stage_rows(seq_base, t0 - TTc, t0, an);
    }
    if (a.dx_in) {
      // <dx_in, X_n> for every stream n
      float w2[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) w2[q] = 0.0f;
      if (tok_ok && lane_ok) {
        float2 gx[4];
        unpack8x2(ld_na(a.dx_in + tok * C + c_lane), gx);
#pragma unroll
        for (int n = 0; n < NMAX; ++n) {
          if (n < N) {
            const int slot = p.is_active[n];
            const __nv_bfloat16* src = slot ? (a.saved_active ? a.saved_active + (tok * k + slot - 1) * C + c_lane
                                                              : a.X + tok * NC + (size_t)n * C + c_lane)
                                            : a.X + tok * NC + (size_t)n * C + c_lane;
            float2 xv[4];
            unpack8x2(ld_na(src), xv);
            w2[n] = dot8(gx, xv);
          }
        }
      }
      const float r = half_transpose_sum16(w2, l16);
      if (tok_ok) st_v(pdot + (tok * ncb + cb) * PDOT + 32 + l16, r);
    }
    if (refill) *reinterpret_cast<uint4*>(&sm.ring[(t0 - TTc - HALO + hw) & (ORc - 1)][8 * l16]) = next_row;
    if (!HAS_CONV) continue;
    __syncthreads();
    // ------------------------------------------------ channel phase
    if (pair_ok) {
      float2 tp[12];
      load_tap_pairs(tp);
      if (has_next) tfa_chunk(tp, t0 - TTc);
      // convolution parts of dout: du rows t0 .. t0 + 18 (rows past the
      // sequence end hold zeros)
      float2 part[TTc];
      if (grp == 0) {
        float2 d1[TTc + 3], d2[TTc + 7];
#pragma unroll
        for (int i = 0; i < TTc + 7; ++i) {
          if (i < TTc + 3) d1[i] = *reinterpret_cast<const float2*>(&sm.du1[(t0 + i) & (col::D1 - 1)][2 * pr]);
          d2[i] = *reinterpret_cast<const float2*>(&sm.du2[(t0 + i) & (col::D2 - 1)][2 * pr]);
        }
#pragma unroll
        for (int tt = 0; tt < TTc; ++tt) part[tt] = __fmul2_rn(tp[0], d1[tt]);
#pragma unroll
        for (int tau = 1; tau < 4; ++tau)
#pragma unroll
          for (int tt = 0; tt < TTc; ++tt) part[tt] = __ffma2_rn(tp[tau], d1[tt + tau], part[tt]);
#pragma unroll
        for (int tau = 0; tau < 8; ++tau)
#pragma unroll
          for (int tt = 0; tt < TTc; ++tt) part[tt] = __ffma2_rn(tp[4 + tau], d2[tt + tau], part[tt]);
        // dw: this chunk's tokens (du of tokens past the end is zero)
        float2 ow[TTc + HALO];
#pragma unroll
        for (int i = 0; i < TTc + HALO; ++i)
          ow[i] = bf2f(*reinterpret_cast<const uint32_t*>(&sm.ring[(t0 - HALO + i) & (ORc - 1)][2 * pr]));
#pragma unroll
        for (int tt = 0; tt < TTc; ++tt) {
#pragma unroll
          for (int tau = 0; tau < 4; ++tau) dw[tau] = __ffma2_rn(d1[tt], ow[tt + HALO - tau], dw[tau]);
#pragma unroll
          for (int tau = 0; tau < 8; ++tau) dw[4 + tau] = __ffma2_rn(d2[tt], ow[tt + HALO - tau], dw[4 + tau]);
        }
      } else {
        float2 d3[TTc + 11];
#pragma unroll
        for (int i = 0; i < TTc + 11; ++i)
          d3[i] = *reinterpret_cast<const float2*>(&sm.du3[(t0 + i) & (col::D3 - 1)][2 * pr]);
#pragma unroll
        for (int tt = 0; tt < TTc; ++tt) part[tt] = __fmul2_rn(tp[0], d3[tt]);
#pragma unroll
        for (int tau = 1; tau < 12; ++tau)
#pragma unroll
          for (int tt = 0; tt < TTc; ++tt) part[tt] = __ffma2_rn(tp[tau], d3[tt + tau], part[tt]);
        float2 ow[TTc + HALO];
#pragma unroll
        for (int i = 0; i < TTc + HALO; ++i)
          ow[i] = bf2f(*reinterpret_cast<const uint32_t*>(&sm.ring[(t0 - HALO + i) & (ORc - 1)][2 * pr]));
#pragma unroll
        for (int tt = 0; tt < TTc; ++tt) {
#pragma unroll
          for (int tau = 0; tau < 12; ++tau) dw[tau] = __ffma2_rn(d3[tt], ow[tt + HALO - tau], dw[tau]);
        }
      }
#pragma unroll
      for (int tt = 0; tt < TTc; ++tt) *reinterpret_cast<float2*>(&sm.dconv[tt][grp][2 * pr]) = part[tt];
    }
    __syncthreads();
    if (!has_next) finalize();                 // the walk ends here: no later token phase
  }
  if (HAS_CONV && pair_ok) {
    float* dst = cpart + (size_t)blockIdx.x * NTAPS * C + c2;
#pragma unroll
    for (int q = 0; q < 12; ++q) {
      float* row = dst + (size_t)(12 * grp + q) * C;
      st_v(row, dw[q].x);
      st_v(row + 1, dw[q].y);
    }
  }
}

// ---------------------------------------------------------------- backward per-token reverse
//
// Half-warp per token (lane e = 4 i + j for H^res entry (i, j)): sums the dot
// partials of every channel block, reruns the Sinkhorn iterations keeping the
// iterates, reverses them, and forms
//   dz  (sigmoid' for H^pre / H^post, Sinkhorn reverse for H^res)
//   dp  = rstd * dz                       -> dP[t][0..63] bf16 hi + lo (zero padded)
//   alpha = <dz, z / rstd> * (-rstd^3 / (N C))   -> rec[t][0]
//   hpre[n]                               -> rec[t][1 + n]

template <bool GS>
__global__ void __launch_bounds__(256) bwd_dz_kernel(Params p, const float* __restrict__ saved,
                                                     const float* __restrict__ pdot, int ncb, int has_dxin,
                                                     __nv_bfloat16* __restrict__ dP, float* __restrict__ rec,
                                                     const float* __restrict__ gsdh, RouterBwd rb, size_t T_all) {
  extern __shared__ float trace_s[];           // [16 tokens][iters][16]: each iteration's column-normalisation input
  const int lane = threadIdx.x & 31, e = lane & 15;
  const int slot = (threadIdx.x >> 5) * 2 + (lane >> 4);
  const size_t t = (size_t)blockIdx.x * 16 + slot;
  const bool live = t < T_all;
  const size_t tc = live ? t : 0;
  const int N = p.N, k = p.k, P = p.P;
  const float* zt = saved + tc * (P + 1);
  const float rstd = zt[P];
  // sums over the channel blocks in block order, eight blocks' loads in flight at a time
  float dres = 0.0f, dpost = 0.0f, dpre = 0.0f;
  const float* pd0 = pdot + tc * ncb * PDOT;
  int c = 0;
  for (; c + 8 <= ncb; c += 8) {
    float a[8], b[8], d[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      a[q] = pd0[(c + q) * PDOT + e];
      b[q] = pd0[(c + q) * PDOT + 16 + e];
      d[q] = has_dxin ? pd0[(c + q) * PDOT + 32 + e] : 0.0f;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      dres += a[q];
      dpost += b[q];
      dpre += d[q];
    }
  }
  for (; c < ncb; ++c) {
    dres += pd0[c * PDOT + e];
    dpost += pd0[c * PDOT + 16 + e];
    if (has_dxin) dpre += pd0[c * PDOT + 32 + e];
  }
  const int i = e >> 2, j = e & 3;
  const bool valid = i < k && j < k;
  const float z = valid ? zt[N + 4 * k + k * i + j] : 0.0f;
  float* tr = trace_s + (size_t)slot * p.iters * 16;
  const float M0 = sinkhorn_init(z, valid);
  float M = M0;
  for (int it = 0; it < p.iters; ++it) M = sinkhorn_step(M, valid, nullptr, &tr[it * 16 + e]);
  float g = valid ? dres : 0.0f;
  for (int it = p.iters - 1; it >= 0; --it) {
    g = norm_reverse_col(g, tr[it * 16 + e], valid);
    // the row normalisation's input: M0, or the previous iteration's output,
    // recomputed from its column-normalisation input by the same operations
    float xr = M0;
    if (it > 0) {
      const float pc = tr[(it - 1) * 16 + e];
      const float s = colsum16(pc);
      xr = valid ? pc * __frcp_rn(s) : 0.0f;
    }
    g = norm_reverse_row(g, xr, valid);
  }
  const float dz_res = valid ? g * M0 : 0.0f;
  float dz_post = 0.0f, dz_pre = 0.0f, hpre = 0.0f;
  const float h = e < 4 * k ? sigmoidf_(zt[N + e]) : 0.0f;
  float dpr = 0.0f, alpha_r = 0.0f, beta_r = 0.0f;   // router: dp of logit e, LayerNorm terms
  if (GS) {
    // dL/dH^post through the Gram-Schmidt fold, from gs_rev_kernel
    if (e < 4 * k) dz_post = gsdh[tc * 16 + e] * h * (1.0f - h);
  } else if (rb.rrec) {
    // Router: a routed slot i >= n_fixed wrote w_i H^post[i] u with w_i its
    // stream's score s; dpost holds D[i][c] = <G_i, u_c> at lane 4 i + c.
    //   dL/dH^post[i][c] = w_i D[i][c];  dL/dw_i = sum_c H^post[i][c] D[i][c]
    //   dL/dr_n = s_n (1 - s_n) dL/dw_i for the routed slot i of stream n
    // r = W_r y, y = (v - m) / sd: the LayerNorm reverse adds, per token,
    //   alpha_r v + beta_r to dL/dv, alpha_r = -(dr . r) / (N C sd^2),
    //   beta_r = -(dr . rs) / (N C sd) - m alpha_r,
    // and dp_r = dr / sd enters the W_r rows of the contractions.
    const int nf = rb.n_fixed;
    const int32_t* ti = rb.tok_idx + tc * k;
    const float* rr = rb.rrec + tc * (2 * N + 2);
    const int si = e >> 2;
    const float w = (e < 4 * k && si >= nf) ? rr[ti[si]] : 1.0f;
    if (e < 4 * k) dz_post = w * dpost * h * (1.0f - h);
    float hd = e < 4 * k ? h * dpost : 0.0f;
    hd += __shfl_xor_sync(FULL, hd, 1);
    hd += __shfl_xor_sync(FULL, hd, 2);            // dL/dw of slot e >> 2
    float dr = 0.0f;
#pragma unroll
    for (int q = 0; q < KMAX; ++q) {
      const float dw_q = __shfl_sync(FULL, hd, (lane & 16) + 4 * q);
      if (q >= nf && q < k && e < N && ti[q] == e) dr += dw_q;
    }
    const float sn = e < N ? rr[e] : 0.0f, rn = e < N ? rr[N + e] : 0.0f;
    const float mean = rr[2 * N], sd = rr[2 * N + 1];
    dr *= sn * (1.0f - sn);
    dpr = dr / sd;
    float a1 = dr * rn, a2 = e < N ? dr * rb.rs[e] : 0.0f;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      a1 += __shfl_xor_sync(FULL, a1, o);
      a2 += __shfl_xor_sync(FULL, a2, o);
    }
    const float ncf = (float)((size_t)N * p.C);
    alpha_r = -a1 / (ncf * sd * sd);
    beta_r = -a2 / (ncf * sd) - mean * alpha_r;
    if (live && e < N) rb.cm[t * N + e] = dpr * mean;
  } else if (e < 4 * k) {
    dz_post = dpost * h * (1.0f - h);
  }
  if (e < N) {
    hpre = sigmoidf_(zt[e]);
    dz_pre = has_dxin ? dpre * hpre * (1.0f - hpre) : 0.0f;
  }
  float part = 0.0f;
  if (e < N) part = fmaf(dz_pre, zt[e], part);
  if (e < 4 * k) part = fmaf(dz_post, zt[N + e], part);
  if (valid) part = fmaf(dz_res, z, part);
  part += __shfl_xor_sync(FULL, part, 1);
  part += __shfl_xor_sync(FULL, part, 2);
  part += __shfl_xor_sync(FULL, part, 4);
  part += __shfl_xor_sync(FULL, part, 8);
  if (!live) return;
  // dp as a bf16 hi part (dP) and lo part (dP + T * 64): hi + lo keeps about
  // 16 bits of dp for the tensor-core contractions
  __nv_bfloat16* dprow = dP + t * 64;
  __nv_bfloat16* dplow = dP + T_all * 64 + t * 64;
  auto put = [&](int q, float v) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    dprow[q] = h;
    dplow[q] = __float2bfloat16_rn(v - __bfloat162float(h));
  };
  if (e < N) put(e, rstd * dz_pre);
  if (e < 4 * k) put(N + e, rstd * dz_post);
  if (valid) put(N + 4 * k + k * i + j, rstd * dz_res);
  // entries P .. P + N - 1: the router logits' dp (zero without a router)
  for (int q = P + e; q < 64; q += 16) put(q, (rb.rrec && q == P + e && e < N) ? dpr : 0.0f);
  const int rl = 1 + N + 4 * k;
  float* rc = rec + t * rl;
  if (e == 0) rc[0] = -part * rstd * rstd / (float)((size_t)N * p.C) + alpha_r;
  if (e == 0 && rb.rrec) rc[1 + N] = beta_r;      // first unused record entry
  if (e < N) rc[1 + e] = hpre;
}

// ---------------------------------------------------------------- Gram-Schmidt reverse
//
// One thread per token.  The write-back used H^post' = H^post T (T: the
// token's Gram-Schmidt coefficients); the column pass's dots give
// D[i][d] = dL/dH^post'[i][d] (summed over the channel blocks here).
//   dL/dH^post[i][c] = sum_d D[i][d] T[c][d]            -> gsdh (read by bwd_dz)
//   dL/dT[c][d]      = sum_i H^post[i][c] D[i][d]
// then back through the Gram-Schmidt steps to dL/dM and S = dM + dM^T, the
// Gram term of dL/du, to sgram (applied by gs_bwd_kernel).

__global__ void __launch_bounds__(64) gs_rev_kernel(Params p, const float* __restrict__ saved,
                                                     const float* __restrict__ pdot, int ncb,
                                                     const float* __restrict__ gsrec, float* __restrict__ gsdh,
                                                     float* __restrict__ sgram, size_t T_all) {
  const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T_all) return;
  float D[KMAX][4];
#pragma unroll
  for (int i = 0; i < KMAX; ++i)
#pragma unroll
    for (int d = 0; d < 4; ++d) D[i][d] = 0.0f;
  const float* pd = pdot + t * ncb * PDOT + 16;
  for (int c = 0; c < ncb; ++c) {
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      const float4 v = *reinterpret_cast<const float4*>(pd + (size_t)c * PDOT + 4 * i);
      D[i][0] += v.x;
      D[i][1] += v.y;
      D[i][2] += v.z;
      D[i][3] += v.w;
    }
  }
  const float* zt = saved + t * (p.P + 1) + p.N;
  float H[KMAX][4];
#pragma unroll
  for (int i = 0; i < KMAX; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      H[i][c] = i < p.k ? sigmoidf_(zt[4 * i + c]) : 0.0f;
      if (i >= p.k) D[i][c] = 0.0f;
    }
  const float* gr = gsrec + t * GS_REC;
  float T[4][4], M[4][4], dT[4][4], dM[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float4 a = *reinterpret_cast<const float4*>(gr + 4 * c);
    const float4 b = *reinterpret_cast<const float4*>(gr + 16 + 4 * c);
    T[c][0] = a.x; T[c][1] = a.y; T[c][2] = a.z; T[c][3] = a.w;
    M[c][0] = b.x; M[c][1] = b.y; M[c][2] = b.z; M[c][3] = b.w;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int d = 0; d < 4; ++d) {
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < KMAX; ++i) s = fmaf(H[i][c], D[i][d], s);
      dT[c][d] = s;
    }
  gs_coeffs_reverse(M, dT, dM);
  float* dh = gsdh + t * 16;
  float* sg = sgram + t * 16;
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    float o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float s = 0.0f;
#pragma unroll
      for (int d = 0; d < 4; ++d) s = fmaf(D[i][d], T[c][d], s);
      o[c] = s;
    }
    *reinterpret_cast<float4*>(dh + 4 * i) = make_float4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<float4*>(sg + 4 * i) =
        make_float4(dM[i][0] + dM[0][i], dM[i][1] + dM[1][i], dM[i][2] + dM[2][i], dM[i][3] + dM[3][i]);
  }
}

cudaError_t launch_gs_rev(const Params& p, const float* saved, const float* pdot, const float* gsrec, float* gsdh,
                          float* sgram, cudaStream_t st) {
  const size_t T_all = (size_t)p.B * p.S;
  const int ncb = (p.C + col::CB - 1) / col::CB;
  timing_begin("gs_rev", st);
  gs_rev_kernel<<<(unsigned)((T_all + 63) / 64), 64, 0, st>>>(p, saved, pdot, ncb, gsrec, gsdh, sgram, T_all);
  timing_end(st);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- launchers

cudaError_t launch_coef(const Params& p, const float* saved, float* coef, cudaStream_t st) {
  const size_t T_all = (size_t)p.B * p.S;
  timing_begin("coef", st);
  coef_kernel<<<(unsigned)((T_all * 16 + 255) / 256), 256, 0, st>>>(p, saved, coef, T_all);
  timing_end(st);
  return cudaGetLastError();
}

bool stream_update_supported(const Params& p) { return p.C % 8 == 0; }

cudaError_t launch_fwd_update(const Params& p, const UpdArgs<__nv_bfloat16>& a, const float* coef, bool has_conv,
                              int sms, cudaStream_t st) {
  const Walk wk = make_walk(p, sms);
  {
    const size_t T = (size_t)p.B * p.S, row = (size_t)p.C * 2;
    dbg::ExtentList l;
    l.add(a.X_in, T * p.N * row).add(a.X_out, T * p.N * row).add(a.out, T * row).add(a.x_in, T * row);
    l.add(a.saved_active, T * p.k * row).add(coef, T * COEF_STRIDE * 4).add(a.tok_idx, T * p.k * 4);
    for (int j = 0; j < 3; ++j) l.add(a.w[j], (size_t)p.C * 4 * (j + 1) * 4);
    if (cudaError_t e = dbg::set_extents(l, st)) return e;
  }
  dim3 grid(wk.R, wk.ncb);
  const int smem = (int)sizeof(FwdSmem);
  timing_begin("fwd_update", st);
  const bool twelve = p.n_inactive == 12;      // N = 16, k = 4
  if (a.tok_idx && has_conv) {
    cudaFuncSetAttribute(fwd_update_kernel<true, -1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    fwd_update_kernel<true, -1><<<grid, THREADS, smem, st>>>(p, a, coef, wk);
  } else if (a.tok_idx) {
    fwd_update_kernel<false, -1><<<grid, THREADS, 0, st>>>(p, a, coef, wk);
  } else if (has_conv && twelve) {
    cudaFuncSetAttribute(fwd_update_kernel<true, 12>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    fwd_update_kernel<true, 12><<<grid, THREADS, smem, st>>>(p, a, coef, wk);
  } else if (has_conv) {
    cudaFuncSetAttribute(fwd_update_kernel<true, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    fwd_update_kernel<true, 0><<<grid, THREADS, smem, st>>>(p, a, coef, wk);
  } else if (twelve) {
    fwd_update_kernel<false, 12><<<grid, THREADS, 0, st>>>(p, a, coef, wk);
  } else {
    fwd_update_kernel<false, 0><<<grid, THREADS, 0, st>>>(p, a, coef, wk);
  }
  timing_end(st);
  return cudaGetLastError();
}

size_t bwd_col_pdot_floats(const Params& p) {
  return (size_t)p.B * p.S * (size_t)((p.C + col::CB - 1) / col::CB) * PDOT;
}
size_t bwd_col_cpart_floats(const Params& p, int sms) {
  return (size_t)make_walk_col(p, sms).R * NTAPS * (size_t)p.C;
}
int bwd_col_cpart_rows(const Params& p, int sms) { return make_walk_col(p, sms).R; }

// Conv weights w4 [C, 4], w8 [C, 8], w12 [C, 12] -> tap-major [24][C]: row g
// is tap g of the three branches in the order of load_taps.
__global__ void col_taps_kernel(const float* __restrict__ w4, const float* __restrict__ w8,
                                const float* __restrict__ w12, float* __restrict__ taps, int C) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= NTAPS * C) return;
  const int g = i / C, c = i - g * C;
  taps[i] = g < 4 ? w4[(size_t)c * 4 + g] : (g < 12 ? w8[(size_t)c * 8 + (g - 4)] : w12[(size_t)c * 12 + (g - 12)]);
}

size_t bwd_col_taps_floats(const Params& p) { return (size_t)NTAPS * p.C; }

cudaError_t launch_bwd_col(const Params& p, const BwdArgs<__nv_bfloat16>& a, const float* coef, bool has_conv,
                           float* pdot, float* cpart, float* taps, int sms, cudaStream_t st) {
  const Walk wk = make_walk_col(p, sms);
  if (has_conv) {
    const int n = NTAPS * p.C;
    timing_begin("col_taps", st);
    col_taps_kernel<<<(n + 255) / 256, 256, 0, st>>>(a.w[0], a.w[1], a.w[2], taps, p.C);
    timing_end(st);
    if (cudaError_t e = cudaGetLastError()) return e;
  }
  {
    const size_t T = (size_t)p.B * p.S, row = (size_t)p.C * 2;
    dbg::ExtentList l;
    l.add(a.X, T * p.N * row).add(a.saved_active, T * p.k * row).add(a.out, T * row).add(a.dXp, T * p.N * row);
    l.add(a.dx_in, T * row).add(a.dX, T * p.N * row).add(a.dout, T * row).add(coef, T * COEF_STRIDE * 4);
    l.add(a.tok_idx, T * p.k * 4).add(pdot, bwd_col_pdot_floats(p) * 4).add(cpart, bwd_col_cpart_floats(p, sms) * 4);
    for (int j = 0; j < 3; ++j) l.add(a.w[j], (size_t)p.C * 4 * (j + 1) * 4);
    if (has_conv) l.add(taps, bwd_col_taps_floats(p) * 4);
    if (cudaError_t e = dbg::set_extents(l, st)) return e;
  }
  dim3 grid(wk.R, wk.ncb);
  const int smem = (int)sizeof(ColSmem);
  timing_begin("bwd_col", st);
  if (has_conv && a.tok_idx) {
    cudaFuncSetAttribute(bwd_col_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    bwd_col_kernel<true, true><<<grid, col::THREADS, smem, st>>>(p, a, coef, pdot, cpart, taps, wk);
  } else if (a.tok_idx) {
    cudaFuncSetAttribute(bwd_col_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    bwd_col_kernel<false, true><<<grid, col::THREADS, smem, st>>>(p, a, coef, pdot, cpart, taps, wk);
  } else if (has_conv) {
    cudaFuncSetAttribute(bwd_col_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    bwd_col_kernel<true, false><<<grid, col::THREADS, smem, st>>>(p, a, coef, pdot, cpart, taps, wk);
  } else {
    cudaFuncSetAttribute(bwd_col_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    bwd_col_kernel<false, false><<<grid, col::THREADS, smem, st>>>(p, a, coef, pdot, cpart, taps, wk);
  }
  timing_end(st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dz(const Params& p, const float* saved, const float* pdot, bool has_dxin,
                          __nv_bfloat16* dP, float* rec, const float* gsdh, const RouterBwd& rb, cudaStream_t st) {
  const size_t T_all = (size_t)p.B * p.S;
  const int ncb = (p.C + col::CB - 1) / col::CB;
  const size_t smem = (size_t)16 * std::max(p.iters, 1) * 16 * sizeof(float);
  const unsigned grid = (unsigned)((T_all + 15) / 16);
  timing_begin("bwd_dz", st);
  if (gsdh) {
    cudaFuncSetAttribute(bwd_dz_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    bwd_dz_kernel<true><<<grid, 256, smem, st>>>(p, saved, pdot, ncb, has_dxin ? 1 : 0, dP, rec, gsdh, rb, T_all);
  } else {
    cudaFuncSetAttribute(bwd_dz_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    bwd_dz_kernel<false><<<grid, 256, smem, st>>>(p, saved, pdot, ncb, has_dxin ? 1 : 0, dP, rec, nullptr, rb,
                                                  T_all);
  }
  timing_end(st);
  return cudaGetLastError();
}

// Reads and clears the first out-of-extent access recorded by a debug build
// (0: none; -1: release build, which records nothing).
int debug_record(unsigned long long* line, unsigned long long* addr) {
#ifdef XHC_DEBUG
  unsigned long long r[2] = {0, 0};
  if (cudaDeviceSynchronize() != cudaSuccess) return -2;
  if (cudaMemcpyFromSymbol(r, dbg::g_record, sizeof(r)) != cudaSuccess) return -2;
  if (line) *line = r[0];
  if (addr) *addr = r[1];
  if (!r[0]) return 0;
  const unsigned long long z[2] = {0, 0};
  cudaMemcpyToSymbol(dbg::g_record, z, sizeof(z));
  return 1;
#else
  if (line) *line = 0;
  if (addr) *addr = 0;
  return -1;
#endif
}

// Debug builds: one checked load outside the registered extent of `buf`
// (`bytes` >= 256 long): the extent covers its first 64 bytes, the load
// targets byte 128, inside the allocation, so even an unchecked load would
// stay in bounds.  The check must skip it and record it.
__global__ void debug_selftest_kernel(const float* buf, float* out) {
  out[0] = ld_f(buf + 32);
}

int debug_selftest(const float* buf, float* out, cudaStream_t st) {
  dbg::ExtentList l;
  l.add(buf, 64).add(out, 4);
  if (dbg::set_extents(l, st) != cudaSuccess) return -2;
  debug_selftest_kernel<<<1, 1, 0, st>>>(buf, out);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

}  // namespace xhc
