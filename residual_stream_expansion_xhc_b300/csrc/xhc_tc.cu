// Tensor-core kernels of the xHC update (sm_103a): tcgen05 MMAs with TMEM
// accumulators fed by TMA.
//
// Method: "xHC: Expanded Hyper-Connections" (qingkeai.online), section
// "Scaling N": the coefficients H^pre, H^post, H^res are generated from the
// whole N*C state of a token; section "Cost of scaling N" notes that this
// projection is the cost that grows with N.  Here it is the one dense
// contraction of the forward: z = rstd * (vec X . W^T), [tokens x N*C] x
// [N*C x P], P = N + 4k + k^2.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "xhc_sm100.cuh"
#include "xhc_bwd.cuh"
#include "xhc_tc.cuh"

namespace xhc {

using namespace sm100;

__device__ int g_device_error = 0;

namespace {
// Failure-detection test hook: when set, the next coefficient projection
// issues no loads (consumed by that launch).
std::atomic<int> g_starve_next_projection{0};
}  // namespace

int set_wait_limit_ns(unsigned long long ns) {
  const unsigned long long v = ns ? ns : 2000000000ull;
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  return cudaMemcpyToSymbol(sm100::g_wait_limit_ns, &v, sizeof(v)) == cudaSuccess ? 0 : -1;
}

void starve_next_projection() { g_starve_next_projection.store(1); }

// ---------------------------------------------------------------- host: tensor maps

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Tiled bf16 tensor map; dims/strides innermost first (strides in bytes, one
// fewer than dims), 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
              const uint32_t* box, CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B,
              CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides[i];
  }
  CUresult r = enc(m, dt, rank, const_cast<void*>(base), d, s, b, e,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

}  // namespace

// ---------------------------------------------------------------- coefficient projection
//
// One CTA per 128-token tile (persistent over tiles).  Warp roles:
//   warp 0      TMA producer: X tile [128 tokens x 64 state entries] and the
//               matching fp32 W tile [P x 64] per stage
//   warp 1      MMA issuer (one thread) and TMEM owner
//   warps 2..9  split the W tile into bf16 W_hi = bf16(W) and W_lo =
//               bf16(W - W_hi) (swizzled K-major tiles), and accumulate the
//               sum of squares of each X stage (warps 2..5 and 6..9 each take
//               half of every token row); warps 2..5 then run the epilogue
//               (rstd, logits, sigmoid, Sinkhorn, stores)
// D[128 x 48] (fp32, TMEM) accumulates X.W_hi^T + X.W_lo^T over all N*C / 64
// stages of a tile, which keeps about 16 mantissa bits of W; two TMEM buffers
// let the epilogue of tile i overlap the MMAs of tile i+1.

namespace coeffs {
constexpr int TILE_T = 128;
constexpr int KC = 64;                  // state entries per stage (128 bytes of bf16)
constexpr int X_BYTES = TILE_T * KC * 2;          // 16 KB (a tile of `rows` <= 128 tokens uses the first rows)
constexpr int W_ROWS = 48;                        // padded P
constexpr int WRAW_BYTES = W_ROWS * KC * 4;       // 12 KB fp32 tile from TMA
constexpr int W_BYTES = W_ROWS * KC * 2;          // 6 KB per bf16 part
constexpr int MATH_WARPS = 8;                     // two per scheduler: W split + sum of squares
constexpr int THREADS = 64 + 32 * MATH_WARPS;     // producer, MMA issuer, math warps
constexpr int TMEM_COLS = 128;                    // 2 buffers x 64 columns
// Stage layouts.  PRESPLIT: W arrives as bf16 hi and lo tiles split once per
// call (w_split_kernel, which stores each stage's 12 KB as one contiguous,
// already swizzled image), so a stage is X + hi + lo.  Otherwise the fp32 W
// tile arrives and the math warps split it into hi and lo in the stage.
// ROUTER: the projection also carries the N router rows W_r (MMA rows 48 ..
// 48 + N - 1, N = 64 columns of the accumulator), for the router's scores.
template <bool PRESPLIT, bool ROUTER = false> struct Layout;
template <> struct Layout<true, false> {
  static constexpr int WR = W_ROWS;                 // rows of W in the MMA
  static constexpr int WPART = W_BYTES;             // bytes of one bf16 part of a 64-column chunk
  static constexpr int BOXES = 2;                   // 64-entry chunks per stage: 256 contiguous bytes per row
  static constexpr int STAGES = 4;
  static constexpr int OFF_WHI = BOXES * X_BYTES;   // chunk b: hi at OFF_WHI + b WBOX, lo WPART later
  static constexpr int OFF_WLO = OFF_WHI + WPART;
  static constexpr int WBOX = 2 * WPART;
  static constexpr int OFF_WRAW = 0;                // unused
  static constexpr int STAGE_BYTES = OFF_WHI + BOXES * WBOX;   // 56 KB
};
template <> struct Layout<false, false> {
  static constexpr int WR = W_ROWS;
  static constexpr int WPART = W_BYTES;
  static constexpr int BOXES = 1;
  static constexpr int WBOX = 0;
  static constexpr int STAGES = 5;
  static constexpr int OFF_WRAW = X_BYTES;
  static constexpr int OFF_WHI = X_BYTES + WRAW_BYTES;
  static constexpr int OFF_WLO = OFF_WHI + W_BYTES;
  static constexpr int STAGE_BYTES = OFF_WLO + W_BYTES;   // 40 KB
};
template <> struct Layout<true, true> {
  static constexpr int WR = 64;
  static constexpr int WPART = WR * KC * 2;         // 8 KB
  static constexpr int BOXES = 2;
  static constexpr int STAGES = 3;
  static constexpr int OFF_WHI = BOXES * X_BYTES;
  static constexpr int OFF_WLO = OFF_WHI + WPART;
  static constexpr int WBOX = 2 * WPART;
  static constexpr int OFF_WRAW = 0;
  static constexpr int STAGE_BYTES = OFF_WHI + BOXES * WBOX;   // 64 KB
};
template <bool PRESPLIT, bool ROUTER = false>
constexpr int smem_bytes() {
  return Layout<PRESPLIT, ROUTER>::STAGES * Layout<PRESPLIT, ROUTER>::STAGE_BYTES + 1024;
}
}  // namespace coeffs

struct CoeffsOut {
  float* hpre;
  float* hpost;
  float* hres;
  float* saved;
  float* coef;    // [T, COEF_STRIDE] coefficient block, or nullptr
  const uint8_t* wsplit;   // stage images of the bf16 hi/lo split of W, or nullptr
  float* router = nullptr; // ROUTER: [T, P + 1] rstd (W_r v) at 0..N-1, rstd sum(v) at N, rstd at P
};

// Sinkhorn of a k x k = 4 x 4 logit block held in registers: the operations
// of sinkhorn_thread in the same order, with every index fixed at compile
// time (so nothing goes through local memory).
__device__ __forceinline__ void sinkhorn4(const float (&z)[16], int iters, float (&M)[4][4]) {
  float zmax = -INFINITY;
#pragma unroll
  for (int e = 0; e < 16; ++e) zmax = fmaxf(zmax, z[e]);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) M[i][j] = expf(z[4 * i + j] - zmax);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float r = __frcp_rn((M[i][0] + M[i][1]) + (M[i][2] + M[i][3]));
#pragma unroll
      for (int j = 0; j < 4; ++j) M[i][j] *= r;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float r = __frcp_rn((M[0][j] + M[1][j]) + (M[2][j] + M[3][j]));
#pragma unroll
      for (int i = 0; i < 4; ++i) M[i][j] *= r;
    }
  }
}

// The epilogue of the N = 16, k = 4 shape split over the two math halves of
// a token row: part 0 the Sinkhorn of H^res (coefficient block entries
// 32..47, and `hres`), part 1 rstd and the logits (`saved`), the sigmoids of
// H^pre and H^post (entries 0..31, `hpre`, `hpost`).  Same values as
// coeffs_epilogue.  The projection's rows are ordered as the coefficient
// block at this shape (P = 48): H^pre 0..15, H^post 16..31, H^res 32..47.
__device__ __forceinline__ void coeffs_epilogue_16x4(const Params& p, const float (&pz)[coeffs::W_ROWS], float ss,
                                                     size_t t, const CoeffsOut& o, int part) {
  const float rstd = 1.0f / sqrtf(ss / (float)(16 * p.C) + p.eps);
  if (part == 0) {
    if (!o.hres && !o.coef) return;
    float z[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) z[e] = rstd * pz[32 + e];
    float M[4][4];
    sinkhorn4(z, p.iters, M);
    if (o.hres) {
      float4* hr = reinterpret_cast<float4*>(o.hres + t * 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) hr[i] = make_float4(M[i][0], M[i][1], M[i][2], M[i][3]);
    }
    if (o.coef) {
      float4* cf = reinterpret_cast<float4*>(o.coef + t * COEF_STRIDE);
#pragma unroll
      for (int i = 0; i < 4; ++i) cf[8 + i] = make_float4(M[i][0], M[i][1], M[i][2], M[i][3]);
    }
    return;
  }
  if (o.saved) {
    float* sv = o.saved + t * 49;
#pragma unroll
    for (int q = 0; q < 48; ++q) sv[q] = rstd * pz[q];
    sv[48] = rstd;
  }
  if (!o.hpre && !o.hpost && !o.coef) return;
  float h[32];
#pragma unroll
  for (int q = 0; q < 32; ++q) h[q] = sigmoidf_(rstd * pz[q]);
  if (o.hpre) {
    float4* d = reinterpret_cast<float4*>(o.hpre + t * 16);
#pragma unroll
    for (int v = 0; v < 4; ++v) d[v] = make_float4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
  }
  if (o.hpost) {
    float4* d = reinterpret_cast<float4*>(o.hpost + t * 16);
#pragma unroll
    for (int v = 0; v < 4; ++v) d[v] = make_float4(h[16 + 4 * v], h[17 + 4 * v], h[18 + 4 * v], h[19 + 4 * v]);
  }
  if (o.coef) {
    float4* cf = reinterpret_cast<float4*>(o.coef + t * COEF_STRIDE);
#pragma unroll
    for (int v = 0; v < 8; ++v) cf[v] = make_float4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
  }
}

// Coefficients of token t from its unscaled logits pz (vec X . W^T) and the
// sum of squares of its state: rstd, logits, sigmoid, Sinkhorn, stores.
__device__ __forceinline__ void coeffs_epilogue(const Params& p, const float (&pz)[coeffs::W_ROWS], float ss,
                                                size_t t, const CoeffsOut& o) {
  const int N = p.N, k = p.k, P = p.P;
  const float rstd = 1.0f / sqrtf(ss / (float)(N * p.C) + p.eps);
  if (o.saved) {
    float* sv = o.saved + t * (P + 1);
#pragma unroll
    for (int q = 0; q < coeffs::W_ROWS; ++q)
      if (q < P) sv[q] = rstd * pz[q];
    sv[P] = rstd;
  }
  float zl[PMAX];
#pragma unroll
  for (int q = 0; q < coeffs::W_ROWS; ++q) zl[q] = rstd * pz[q];
  if (o.hpre) {
#pragma unroll
    for (int q = 0; q < NMAX; ++q)
      if (q < N) o.hpre[t * N + q] = sigmoidf_(zl[q]);
  }
  if (o.hpost) {
#pragma unroll
    for (int q = 0; q < 4 * KMAX; ++q)
      if (q < 4 * k) o.hpost[t * 4 * k + q] = sigmoidf_(zl[N + q]);
  }
  if (o.hres || o.coef) {
    // Sinkhorn of this token's k x k logits in registers (one thread)
    float M[KMAX][KMAX];
    sinkhorn_thread(zl + N + 4 * k, k, p.iters, M);
    if (o.hres) {
#pragma unroll
      for (int i = 0; i < KMAX; ++i)
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (i < k && j < k) o.hres[t * k * k + k * i + j] = M[i][j];
    }
    if (o.coef) {
      float4* cf = reinterpret_cast<float4*>(o.coef + t * COEF_STRIDE);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        float h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = (4 * v + e < N) ? sigmoidf_(zl[4 * v + e]) : 0.0f;
        cf[v] = make_float4(h[0], h[1], h[2], h[3]);
      }
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        float h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = (4 * v + e < 4 * k) ? sigmoidf_(zl[N + 4 * v + e]) : 0.0f;
        cf[4 + v] = make_float4(h[0], h[1], h[2], h[3]);
      }
#pragma unroll
      for (int i = 0; i < KMAX; ++i) cf[8 + i] = make_float4(M[i][0], M[i][1], M[i][2], M[i][3]);
    }
  }
}

template <bool PRESPLIT, bool ROUTER>
__global__ void __launch_bounds__(coeffs::THREADS, 1)
    coeffs_tc_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapW,
                     const __grid_constant__ CUtensorMap mapWlo, Params p, CoeffsOut o, int ntiles, int rows,
                     int starve) {
  using namespace coeffs;
  using L = Layout<PRESPLIT, ROUTER>;
  constexpr int STAGES = L::STAGES, STAGE_BYTES = L::STAGE_BYTES, BOXES = L::BOXES;
  constexpr int OFF_WRAW = L::OFF_WRAW, OFF_WHI = L::OFF_WHI, OFF_WLO = L::OFF_WLO;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint64_t full[STAGES], bready[STAGES], empty[STAGES], tfull[2], tempty[2], ssfull[2], ssempty[2],
      mdrain;
  __shared__ uint32_t tmem_slot;
  __shared__ float ss_half[2][TILE_T];          // the two halves' row sums of squares
  __shared__ float s1_half[ROUTER ? 2 : 1][ROUTER ? TILE_T : 1];   // ROUTER: and their row sums
  int* err = &g_device_error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cchunks = p.C / (KC * BOXES);
  const int nk = p.N * cchunks;                 // stages per tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);                   // TMA transaction
      mbar_init(&bready[s], MATH_WARPS);        // W split done by the math warps
      mbar_init(&empty[s], 1 + MATH_WARPS);     // MMA commit + the math warps done reading X
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], MATH_WARPS);        // every math warp (those that do not read it arrive at once)
      mbar_init(&ssfull[b], MATH_WARPS);        // both halves wrote their row sums (index 0 used)
      mbar_init(&ssempty[b], MATH_WARPS);       // and read them
    }
    mbar_init(&mdrain, 1);                      // every MMA of the CTA complete
    fence_mbar_init();
    tma_prefetch_desc(&mapX);
    if (!PRESPLIT) tma_prefetch_desc(&mapW);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_first(), pol_w = policy_evict_last();
      int it = 0;
      if (starve) goto done_prod;               // test hook: no loads, so every consumer's wait runs out
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        for (int kc = 0; kc < nk; ++kc, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (it >= STAGES && !mbar_wait(&empty[s], ph ^ 1, err, 11)) goto done_prod;
          uint8_t* st = smem + s * STAGE_BYTES;
          mbar_expect_tx(&full[s], BOXES * rows * KC * 2 + (PRESPLIT ? BOXES * 2 * L::WPART : p.P * KC * 4));
          const int n = kc / cchunks, c0 = (kc % cchunks) * KC * BOXES;
#pragma unroll
          for (int b = 0; b < BOXES; ++b) tma_load_3d(st + b * X_BYTES, &mapX, &full[s], c0 + b * KC, n, tile * rows, pol_x);
          if (PRESPLIT) {
            bulk_load(st + OFF_WHI, o.wsplit + (size_t)kc * BOXES * 2 * L::WPART, BOXES * 2 * L::WPART, &full[s],
                      pol_w);
          } else {
            tma_load_2d_f32(st + OFF_WRAW, &mapW, &full[s], kc * KC, 0, pol_w);
          }
        }
      }
    done_prod:
      // the loads issued land before the CTA may end (on every path: after
      // a normal run these waits return at once)
      for (int d = it > STAGES ? it - STAGES : 0; d < it; ++d) mbar_wait_drain(&full[d % STAGES], (d / STAGES) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(TILE_T, L::WR, 0, 0);
      int it = 0, tl = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tl) {
        const int buf = tl & 1;
        if (tl >= 2 && !mbar_wait(&tempty[buf], ((tl >> 1) & 1) ^ 1, err, 12)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * 64;
        bool ok = true;
        for (int kc = 0; kc < nk; ++kc, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(PRESPLIT ? &full[s] : &bready[s], (it / STAGES) & 1, err, 13)) { ok = false; break; }
          tc_fence_after();
          const uint32_t xs = smem_u32(smem + s * STAGE_BYTES);
#pragma unroll
          for (int b = 0; b < BOXES; ++b) {
#pragma unroll
            for (int ks = 0; ks < KC / 16; ++ks) {
              const uint64_t a = sdesc_sw128(xs + b * X_BYTES + ks * 32, 16, 1024);
              const uint64_t bh = sdesc_sw128(xs + OFF_WHI + b * L::WBOX + ks * 32, 16, 1024);
              const uint64_t bl = sdesc_sw128(xs + OFF_WLO + b * L::WBOX + ks * 32, 16, 1024);
              umma_bf16(d, a, bh, idesc, (kc | b | ks) != 0);
              umma_bf16(d, a, bl, idesc, 1);
            }
          }
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&tfull[buf]);
      }
      // every MMA issued completes before the CTA may end
      umma_commit(&mdrain);
      mbar_wait_drain(&mdrain, 0);
    }
  } else {
    // ------------------------------------------------ sum of squares + epilogue
    const int row = 32 * (warp & 3) + lane;             // token row == TMEM lane
    const int half = (warp - 2) >> 2;                   // which four 16-byte chunks of the row
    const int mt = threadIdx.x - 64;                    // math thread 0 .. 32 * MATH_WARPS - 1
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    int it = 0, tl = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tl) {
      float ss = 0.0f, s1 = 0.0f;
      bool ok = true;
      for (int kc = 0; kc < nk; ++kc, ++it) {
        const int s = it % STAGES;
        if (!mbar_wait(&full[s], (it / STAGES) & 1, err, 14)) { ok = false; break; }
        uint8_t* stg = smem + s * STAGE_BYTES;
        // split W: 48 rows x 8 groups of 8 entries over the math threads
        for (int u = mt; !PRESPLIT && u < W_ROWS * 8; u += 32 * MATH_WARPS) {
          const int q = u >> 3, g = u & 7;
          uint4 h = make_uint4(0, 0, 0, 0), l = make_uint4(0, 0, 0, 0);
          if (q < p.P) {
            const float4 a = *reinterpret_cast<const float4*>(stg + OFF_WRAW + q * 256 + g * 32);
            const float4 b = *reinterpret_cast<const float4*>(stg + OFF_WRAW + q * 256 + g * 32 + 16);
            const float w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t hh[4], ll[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat16 h0 = __float2bfloat16_rn(w[2 * e]), h1 = __float2bfloat16_rn(w[2 * e + 1]);
              const float r0 = w[2 * e] - __bfloat162float(h0), r1 = w[2 * e + 1] - __bfloat162float(h1);
              hh[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
              ll[e] = pack_bf2(r0, r1);
            }
            h = make_uint4(hh[0], hh[1], hh[2], hh[3]);
            l = make_uint4(ll[0], ll[1], ll[2], ll[3]);
          }
          *reinterpret_cast<uint4*>(stg + OFF_WHI + sw128_offset(q, g * 16)) = h;
          *reinterpret_cast<uint4*>(stg + OFF_WLO + sw128_offset(q, g * 16)) = l;
        }
        if (!PRESPLIT) {
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bready[s]);   // the MMA may start; X is read below
        }
#pragma unroll
        for (int c = 0; c < 4 * BOXES; ++c) {
          // the row's 8 BOXES 16-byte groups, half of them per math half;
          // physical group (lin + row) mod 8 of box lin / 8: the eight rows
          // read by a phase of eight lanes fall in eight different bank groups
          const int lin = half * 4 * BOXES + c;
          const uint8_t* xr = stg + (lin >> 3) * X_BYTES + row * 128;
          const uint4 v = *reinterpret_cast<const uint4*>(xr + 16 * ((lin + row) & 7));
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float a = bf_lo(w[h]), b = bf_hi(w[h]);
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
            if (ROUTER) s1 += a + b;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      if (!ok) break;
      // the row's total sum of squares from both halves (the same sum, in
      // the same order, in both)
      if (tl >= 1 && !mbar_wait(&ssempty[0], (tl - 1) & 1, err, 16)) break;
      ss_half[half][row] = ss;
      if (ROUTER) s1_half[half][row] = s1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ssfull[0]);
      if (!mbar_wait(&ssfull[0], tl & 1, err, 17)) break;
      ss = ss_half[0][row] + ss_half[1][row];
      if (ROUTER) s1 = s1_half[0][row] + s1_half[1][row];
      __syncwarp();
      if (lane == 0) mbar_arrive(&ssempty[0]);
      // at N = 16, k = 4 both halves share the epilogue; otherwise half 0 alone
      const bool split = p.N == 16 && p.k == 4;
      const int buf = tl & 1;
      if (!split && half == 1) {
        if (lane == 0) mbar_arrive(&tempty[buf]);
        continue;
      }
      if (!mbar_wait(&tfull[buf], (tl >> 1) & 1, err, 15)) break;
      tc_fence_after();
      float pz[L::WR];
#pragma unroll
      for (int c = 0; c < L::WR; c += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + buf * 64 + c, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) pz[c + j] = __uint_as_float(r[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);

      const size_t t = (size_t)tile * rows + row;
      if (row >= rows || t >= (size_t)p.B * p.S) continue;
      const float (&pzc)[W_ROWS] = *reinterpret_cast<const float(*)[W_ROWS]>(&pz[0]);
      if (split) coeffs_epilogue_16x4(p, pzc, ss, t, o, half);
      else coeffs_epilogue(p, pzc, ss, t, o);
      if (ROUTER && half == 0) {
        // the router's logits and the LayerNorm's sum, scaled by rstd
        const float rstd = 1.0f / sqrtf(ss / (float)(p.N * p.C) + p.eps);
        float* zr = o.router + t * (p.P + 1);
#pragma unroll
        for (int n = 0; n < NMAX; ++n)
          if (n < p.N) zr[n] = rstd * pz[W_ROWS + n];
        zr[p.N] = rstd * s1;
        zr[p.P] = rstd;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------- fused stack step
//
// One pass over the state per sublayer of a stack (section "Beyond N=16":
// xHC-Flash lowers a sublayer's traffic by reordering reads and writes across
// sublayers).  For sublayer l the pass
//   - reads every stream of S_l once (TMA tiles [128 tokens x 64 channels]),
//   - forms the dense read x_in_l = sum_n hpre_l[n] S_l[n] (section "Dense
//     read, sparse write"),
//   - rewrites the k active rows of each tile in shared memory with the
//     update of sublayer l (H^res mix + H^post of the TFA components) and
//     stores them back in place (TMA stores),
//   - and projects the tile, as it now holds S_{l+1}, onto W_{l+1} on the
//     tensor cores (bf16 hi + lo parts of W, fp32 TMEM accumulators), with the
//     sum of squares taken on the same values,
// so that the epilogue writes sublayer l+1's coefficient block: the separate
// coefficient pass over S_{l+1} (16 C of reads per token) disappears, and a
// sublayer of the stack costs the update pass's 22 C.
//
// Stage order within a 64-channel chunk: the k active streams of sublayer l
// first (slot order), then the others.  Warp roles as in the coefficient
// pass: warp 0 TMA producer (state tiles, W_{l+1} image, the chunk's `out`
// tile with 16 rows of history and its tap-major conv weights), warp 1 MMA
// issuer, warps 2..9 math (two threads per token row, 32 channels each):
// dense read, update, sum of squares, then the epilogue; warp 10 stores the
// rewritten active tiles (TMA) and releases their stages once the stores
// have read them, on behalf of the math warps, which go straight on to the
// other streams.
namespace flash {
constexpr int TILE_T = 128;
constexpr int KC = 64;
constexpr int X_BYTES = TILE_T * KC * 2;                 // 16 KB
constexpr int W_BYTES = coeffs::W_BYTES;                 // 6 KB per bf16 part
constexpr int STAGE_BYTES = X_BYTES + 2 * W_BYTES;       // 28 KB
constexpr int STAGES = 7;
constexpr int HALO_R = 16;               // out rows above the tile (11 used; 16 keeps the swizzle phase of row r)
constexpr int OUT_BYTES = (TILE_T + HALO_R) * 128;       // 18 KB
constexpr int TAP_BYTES = NTAPS * KC * 4;                // [24 taps][64 channels] fp32
constexpr int OFF_OUT = STAGES * STAGE_BYTES;
constexpr int OFF_TAP = OFF_OUT + OUT_BYTES;
constexpr int SMEM = OFF_TAP + TAP_BYTES + 1024;
constexpr int MATH_WARPS = 8;
constexpr int STORE_WARP = 2 + MATH_WARPS;
constexpr int THREADS = 64 + 32 * MATH_WARPS + 32;
constexpr int TMEM_COLS = 128;
}  // namespace flash

struct FlashArgs {
  const float* coef;       // [T, COEF_STRIDE] coefficients of sublayer l
  const float* taps;       // tap-major conv weights of sublayer l ([C/64][24][64]) or nullptr
  const uint8_t* wsplit;   // stage images of the hi/lo split of W_{l+1}
  __nv_bfloat16* x_in;     // [T, C] or nullptr
  CoeffsOut next;          // sublayer l+1: coef block and saved logits
};

template <bool HAS_CONV>
__global__ void __launch_bounds__(flash::THREADS, 1)
    flash_tc_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapOut, Params p,
                    FlashArgs f, int ntiles, int rows) {
  using namespace flash;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint64_t full[STAGES], bready[STAGES], empty[STAGES], ofull, oempty, updated, tfull[2], tempty[2],
      ssfull[2], ssempty[2], mdrain;
  __shared__ uint32_t tmem_slot;
  __shared__ int ord[NMAX];
  __shared__ float ss_half[2][TILE_T];
  int* err = &g_device_error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, k = p.k, C = p.C;
  const int cchunks = C / KC;
  const size_t T_all = (size_t)p.B * p.S;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&bready[s], MATH_WARPS);       // stage seen (inactive) or rewritten (active) by every math warp
      mbar_init(&empty[s], 1 + MATH_WARPS);    // MMA commit + the math warps
    }
    mbar_init(&ofull, 1);
    mbar_init(&oempty, MATH_WARPS);
    mbar_init(&updated, MATH_WARPS);           // the chunk's active rows rewritten by every math warp
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], MATH_WARPS);
      mbar_init(&ssfull[b], MATH_WARPS);
      mbar_init(&ssempty[b], MATH_WARPS);
    }
    mbar_init(&mdrain, 1);
    for (int i = 0; i < k; ++i) ord[i] = p.idx[i];
    for (int j = 0; j < N - k; ++j) ord[k + j] = p.inactive[j];
    fence_mbar_init();
    tma_prefetch_desc(&mapX);
    tma_prefetch_desc(&mapOut);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_first(), pol_w = policy_evict_last();
      int it = 0, oc = 0, nout = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        for (int cc = 0; cc < cchunks; ++cc, ++oc) {
          if (oc > 0 && !mbar_wait(&oempty, (oc - 1) & 1, err, 21)) goto done_prod;
          ++nout;
          mbar_expect_tx(&ofull, (rows + HALO_R) * 128 + (HAS_CONV ? TAP_BYTES : 0));
          tma_load_2d(smem + OFF_OUT, &mapOut, &ofull, cc * KC, tile * rows - HALO_R, pol_x);
          if (HAS_CONV) bulk_load(smem + OFF_TAP, f.taps + (size_t)cc * NTAPS * KC, TAP_BYTES, &ofull, pol_w);
          for (int j = 0; j < N; ++j, ++it) {
            const int s = it % STAGES;
            if (it >= STAGES && !mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, err, 22)) goto done_prod;
            uint8_t* st = smem + s * STAGE_BYTES;
            const int n = ord[j];
            mbar_expect_tx(&full[s], rows * KC * 2 + 2 * W_BYTES);
            tma_load_3d(st, &mapX, &full[s], cc * KC, n, tile * rows, pol_x);
            bulk_load(st + X_BYTES, f.wsplit + (size_t)(n * cchunks + cc) * 2 * W_BYTES, 2 * W_BYTES, &full[s],
                      pol_w);
          }
        }
      }
    done_prod:
      // the loads issued land before the CTA may end
      for (int d = it > STAGES ? it - STAGES : 0; d < it; ++d) mbar_wait_drain(&full[d % STAGES], (d / STAGES) & 1);
      if (nout > 0) mbar_wait_drain(&ofull, (nout - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(TILE_T, coeffs::W_ROWS, 0, 0);
      int it = 0, tl = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tl) {
        const int buf = tl & 1;
        if (tl >= 2 && !mbar_wait(&tempty[buf], ((tl >> 1) & 1) ^ 1, err, 23)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * 64;
        bool ok = true;
        for (int kc = 0; kc < cchunks * N; ++kc, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&bready[s], (it / STAGES) & 1, err, 24)) { ok = false; break; }
          tc_fence_after();
          const uint32_t xs = smem_u32(smem + s * STAGE_BYTES);
#pragma unroll
          for (int ks = 0; ks < KC / 16; ++ks) {
            const uint64_t a = sdesc_sw128(xs + ks * 32, 16, 1024);
            const uint64_t bh = sdesc_sw128(xs + X_BYTES + ks * 32, 16, 1024);
            const uint64_t bl = sdesc_sw128(xs + X_BYTES + W_BYTES + ks * 32, 16, 1024);
            umma_bf16(d, a, bh, idesc, (kc | ks) != 0);
            umma_bf16(d, a, bl, idesc, 1);
          }
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&tfull[buf]);
      }
      umma_commit(&mdrain);
      mbar_wait_drain(&mdrain, 0);
    }
  } else if (warp == STORE_WARP) {
    // ------------------------------------------------ active tile stores
    if (lane == 0) {
      int it = 0, oc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
        for (int cc = 0; cc < cchunks; ++cc, ++oc, it += N) {
          // every math warp has rewritten its rows of the chunk's k active tiles
          if (!mbar_wait(&updated, oc & 1, err, 31)) { ok = false; break; }
          for (int i = 0; i < k; ++i)
            tma_store_3d(&mapX, smem + ((it + i) % STAGES) * STAGE_BYTES, cc * KC, ord[i], tile * rows);
          tma_store_commit();
          tma_store_wait_read0();
          // the math warps' releases of these stages (the MMA commits its own)
          for (int i = 0; i < k; ++i) mbar_arrive_cnt(&empty[(it + i) % STAGES], MATH_WARPS);
        }
      }
      tma_store_wait0();
    }
  } else {
    // ------------------------------------------------ math: dense read, update, sum of squares, epilogue
    const int row = 32 * (warp & 3) + lane;             // token row == TMEM lane
    const int half = (warp - 2) >> 2;                   // channels 32 half .. 32 half + 31 of each chunk
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    int it = 0, tl = 0, oc = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tl) {
      const size_t t = (size_t)tile * rows + row;
      const bool live = row < rows && t < T_all;
      const float* cf = f.coef + (live ? t : 0) * COEF_STRIDE;
      float hpost[KMAX][4], hres[KMAX][KMAX], hact[KMAX];
#pragma unroll
      for (int i = 0; i < KMAX; ++i) {
        const float4 a = *reinterpret_cast<const float4*>(cf + COEF_POST + 4 * i);
        const float4 b = *reinterpret_cast<const float4*>(cf + COEF_RES + 4 * i);
        hpost[i][0] = a.x; hpost[i][1] = a.y; hpost[i][2] = a.z; hpost[i][3] = a.w;
        hres[i][0] = b.x; hres[i][1] = b.y; hres[i][2] = b.z; hres[i][3] = b.w;
        hact[i] = i < k ? cf[ord[i]] : 0.0f;
      }
      const int spos = live ? (int)(t % (size_t)p.S) : 0;
      float ss = 0.0f;
      bool ok = true;
      for (int cc = 0; cc < cchunks; ++cc, ++oc) {
        float xacc[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) xacc[e] = 0.0f;
        if (!mbar_wait(&ofull, oc & 1, err, 25)) { ok = false; break; }
        // ---- the k active rows of this chunk: read, update, write back
#pragma unroll
        for (int i = 0; i < KMAX; ++i)
          if (i < k && !mbar_wait(&full[(it + i) % STAGES], ((it + i) / STAGES) & 1, err, 26)) ok = false;
        if (!ok) break;
        const uint8_t* os = smem + OFF_OUT;
        const float* tp = reinterpret_cast<const float*>(smem + OFF_TAP);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int gl = half * 4 + q;                    // 16-byte group of the row (8 channels)
          const uint32_t off = row * 128 + ((gl ^ (row & 7)) << 4);
          // channel pairs (2e, 2e + 1) in fp32x2: each lane is the scalar
          // fmaf of that channel, in the same order
          float2 o[KMAX][4];
#pragma unroll
          for (int i = 0; i < KMAX; ++i) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (i < k) v = *reinterpret_cast<const uint4*>(smem + ((it + i) % STAGES) * STAGE_BYTES + off);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) o[i][e] = make_float2(bf_lo(w[e]), bf_hi(w[e]));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float2 xa = make_float2(xacc[8 * q + 2 * e], xacc[8 * q + 2 * e + 1]);
              xa = __ffma2_rn(make_float2(hact[i], hact[i]), o[i][e], xa);
              xacc[8 * q + 2 * e] = xa.x;
              xacc[8 * q + 2 * e + 1] = xa.y;
            }
          }
          // TFA components of this token's 8 channels; row r of the tile is
          // row r + HALO_R of the out tile, tap tau reads row r + HALO_R - tau
          float2 u[4][4];
          {
            const uint4 v = *reinterpret_cast<const uint4*>(os + (row + HALO_R) * 128 + ((gl ^ (row & 7)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) u[0][e] = make_float2(bf_lo(w[e]), bf_hi(w[e]));
          }
#pragma unroll
          for (int c = 1; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) u[c][e] = make_float2(0.0f, 0.0f);
          if (HAS_CONV) {
#pragma unroll
            for (int tau = 0; tau < 12; ++tau) {
              const int r = row + HALO_R - tau;
              uint4 v = *reinterpret_cast<const uint4*>(os + r * 128 + ((gl ^ (r & 7)) << 4));
              if (tau > spos) v = make_uint4(0, 0, 0, 0);   // before the start of the sequence
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
              float2 x[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) x[e] = make_float2(bf_lo(w[e]), bf_hi(w[e]));
              // tap rows: w4 taps at rows 0..3, w8 at 4..11, w12 at 12..23
#pragma unroll
              for (int c = 1; c < 4; ++c) {
                const int K = 4 * c, r0 = (c == 1) ? 0 : (c == 2 ? 4 : 12);
                if (tau < K) {
                  const float4 a = *reinterpret_cast<const float4*>(tp + (r0 + tau) * KC + gl * 8);
                  const float4 b = *reinterpret_cast<const float4*>(tp + (r0 + tau) * KC + gl * 8 + 4);
                  u[c][0] = __ffma2_rn(make_float2(a.x, a.y), x[0], u[c][0]);
                  u[c][1] = __ffma2_rn(make_float2(a.z, a.w), x[1], u[c][1]);
                  u[c][2] = __ffma2_rn(make_float2(b.x, b.y), x[2], u[c][2]);
                  u[c][3] = __ffma2_rn(make_float2(b.z, b.w), x[3], u[c][3]);
                }
              }
            }
          }
          // the new active rows: X'[a_i] = sum_j Hres[i][j] X[a_j] + sum_c Hpost[i][c] u_c
#pragma unroll
          for (int i = 0; i < KMAX; ++i) {
            if (i < k) {
              float2 y[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < KMAX; ++j) acc = __ffma2_rn(make_float2(hres[i][j], hres[i][j]), o[j][e], acc);
#pragma unroll
                for (int c = 0; c < 4; ++c) acc = __ffma2_rn(make_float2(hpost[i][c], hpost[i][c]), u[c][e], acc);
                y[e] = acc;
              }
              uint4 v;
              v.x = pack_bf2(y[0].x, y[0].y);
              v.y = pack_bf2(y[1].x, y[1].y);
              v.z = pack_bf2(y[2].x, y[2].y);
              v.w = pack_bf2(y[3].x, y[3].y);
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float a = bf_lo(w[e]), b = bf_hi(w[e]);
                ss = fmaf(a, a, ss);
                ss = fmaf(b, b, ss);
              }
              if (live) *reinterpret_cast<uint4*>(smem + ((it + i) % STAGES) * STAGE_BYTES + off) = v;
            }
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int i = 0; i < k; ++i) mbar_arrive(&bready[(it + i) % STAGES]);
          mbar_arrive(&oempty);
          mbar_arrive(&updated);          // the store warp stores the rows and releases the stages
        }
        it += k;
        // ---- the other streams: dense read and sum of squares
        for (int j = k; j < N; ++j, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&full[s], (it / STAGES) & 1, err, 27)) { ok = false; break; }
          if (lane == 0) mbar_arrive(&bready[s]);
          const float h = cf[ord[j]];
          const uint8_t* xs = smem + s * STAGE_BYTES + row * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int gl = half * 4 + q;
            const uint4 v = *reinterpret_cast<const uint4*>(xs + ((gl ^ (row & 7)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a = bf_lo(w[e]), b = bf_hi(w[e]);
              ss = fmaf(a, a, ss);
              ss = fmaf(b, b, ss);
              const float2 xa = __ffma2_rn(make_float2(h, h), make_float2(a, b),
                                           make_float2(xacc[8 * q + 2 * e], xacc[8 * q + 2 * e + 1]));
              xacc[8 * q + 2 * e] = xa.x;
              xacc[8 * q + 2 * e + 1] = xa.y;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (!ok) break;
        if (f.x_in && live) {
          uint4* dst = reinterpret_cast<uint4*>(f.x_in + t * C + cc * KC + half * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(pack_bf2(xacc[8 * q], xacc[8 * q + 1]), pack_bf2(xacc[8 * q + 2], xacc[8 * q + 3]),
                                pack_bf2(xacc[8 * q + 4], xacc[8 * q + 5]),
                                pack_bf2(xacc[8 * q + 6], xacc[8 * q + 7]));
        }
      }
      if (!ok) break;
      // ---- epilogue: sublayer l+1's coefficients from the projection of S_{l+1}
      if (tl >= 1 && !mbar_wait(&ssempty[0], (tl - 1) & 1, err, 28)) break;
      ss_half[half][row] = ss;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ssfull[0]);
      if (!mbar_wait(&ssfull[0], tl & 1, err, 29)) break;
      ss = ss_half[0][row] + ss_half[1][row];
      __syncwarp();
      if (lane == 0) mbar_arrive(&ssempty[0]);
      // half 0 runs the epilogue (the split one of the projection would cost
      // this kernel spills: it holds more registers through the chunk loop)
      const int buf = tl & 1;
      if (half == 1) {
        if (lane == 0) mbar_arrive(&tempty[buf]);
        continue;
      }
      if (!mbar_wait(&tfull[buf], (tl >> 1) & 1, err, 30)) break;
      tc_fence_after();
      float pz[coeffs::W_ROWS];
#pragma unroll
      for (int c = 0; c < coeffs::W_ROWS; c += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + buf * 64 + c, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) pz[c + j] = __uint_as_float(r[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      if (live) coeffs_epilogue(p, pz, ss, t, f.next);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------- launchers

bool tc_coeffs_supported(const Params& p) { return p.C % coeffs::KC == 0 && p.P <= coeffs::W_ROWS; }

// W [P, N*C] fp32 -> bf16 hi and lo parts (rows >= P zero), stored tile by
// tile in the exact shared-memory image a stage of the projection needs: for
// each 64-column chunk kk, [hi: 48 rows x 128 B][lo: 48 rows x 128 B], each
// row's eight 16-byte groups placed by the 128-byte swizzle (group g of row q
// at (g ^ (q mod 8)) * 16).  One bulk copy then brings a stage's 12 KB.  One
// thread per 8 consecutive columns of one row.
// With Wr (the router): `rows` = 64, rows 48 .. 48 + NR - 1 of the image are
// the rows of Wr.
__global__ void w_split_kernel(const float* __restrict__ W, uint8_t* __restrict__ Ws, int P, size_t NC,
                               const float* __restrict__ Wr = nullptr, int NR = 0, int rows = coeffs::W_ROWS) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t groups = NC / 8;
  if (i >= (size_t)rows * groups) return;
  const int q = (int)(i / groups);
  const size_t c = (i % groups) * 8;
  float w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const float* src = q < P ? W + (size_t)q * NC
                           : (Wr && q >= coeffs::W_ROWS && q < coeffs::W_ROWS + NR ? Wr + (size_t)(q - coeffs::W_ROWS) * NC
                                                                                    : nullptr);
  if (src) {
    const float4 a = *reinterpret_cast<const float4*>(src + c);
    const float4 b = *reinterpret_cast<const float4*>(src + c + 4);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    h[e] = pack_bf2(w[2 * e], w[2 * e + 1]);
    l[e] = pack_bf2(w[2 * e] - bf_lo(h[e]), w[2 * e + 1] - bf_hi(h[e]));
  }
  const size_t kk = c / coeffs::KC;
  const int g = (int)((c % coeffs::KC) / 8);
  const size_t part = (size_t)rows * coeffs::KC * 2;
  uint8_t* tile = Ws + kk * 2 * part;
  const uint32_t off = sw128_offset(q, g * 16);
  *reinterpret_cast<uint4*>(tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(tile + part + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

size_t coeffs_wsplit_bytes(const Params& p) { return (size_t)2 * coeffs::W_ROWS * p.N * p.C * sizeof(uint16_t); }

cudaError_t launch_coeffs_tc(const Params& p, const void* X, const float* W, void* Wsplit, float* hpre,
                             float* hpost, float* hres, float* saved, float* coef, cudaStream_t st) {
  using namespace coeffs;
  const size_t T_all = (size_t)p.B * p.S;
  const size_t NC = (size_t)p.N * p.C;
  // Tokens per tile: spread the tokens over every SM in one wave where that
  // keeps at least 64 tokens per tile (W is re-read from L2 once per tile);
  // the MMA always computes 128 rows and rows >= `rows` are ignored.
  const size_t per_sm = (T_all + sm_count() - 1) / sm_count();
  const int rows = (int)std::min<size_t>(TILE_T, std::max<size_t>(64, (per_sm + 7) / 8 * 8));
  CUtensorMap mx, mw, mwl;
  {
    const uint64_t dims[3] = {(uint64_t)p.C, (uint64_t)p.N, T_all};
    const uint64_t strides[2] = {(uint64_t)p.C * 2, NC * 2};
    const uint32_t box[3] = {KC, 1, (uint32_t)rows};
    if (!make_map(&mx, X, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const bool presplit = Wsplit != nullptr && p.C % (KC * Layout<true>::BOXES) == 0;
  if (presplit) {
    mw = mx;                                    // unused: W comes by bulk copies
    mwl = mx;
  } else {
    const uint64_t dims[2] = {NC, (uint64_t)p.P};
    const uint64_t strides[1] = {NC * 4};
    const uint32_t box[2] = {KC, (uint32_t)p.P};
    if (!make_map(&mw, W, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return cudaErrorInvalidValue;
    mwl = mw;
  }
  const int ntiles = (int)((T_all + rows - 1) / rows);
  const int grid = std::min(ntiles, sm_count());
  CoeffsOut o{hpre, hpost, hres, saved, coef, (const uint8_t*)Wsplit};
  const int starve = g_starve_next_projection.exchange(0);
  if (presplit) {
    const size_t threads = (size_t)W_ROWS * (NC / 8);
    timing_begin("w_split", st);
    w_split_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(W, (uint8_t*)Wsplit, p.P, NC);
    timing_end(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaFuncSetAttribute(coeffs_tc_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         smem_bytes<true>());
    timing_begin("coeffs_tc", st);
    coeffs_tc_kernel<true, false><<<grid, THREADS, smem_bytes<true>(), st>>>(mx, mw, mwl, p, o, ntiles, rows, starve);
  } else {
    cudaFuncSetAttribute(coeffs_tc_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         smem_bytes<false>());
    timing_begin("coeffs_tc", st);
    coeffs_tc_kernel<false, false><<<grid, THREADS, smem_bytes<false>(), st>>>(mx, mw, mwl, p, o, ntiles, rows,
                                                                              starve);
  }
  timing_end(st);
  return cudaGetLastError();
}

size_t coeffs_router_wsplit_bytes(const Params& p) {
  return (size_t)2 * coeffs::Layout<true, true>::WR * p.N * p.C * sizeof(uint16_t);
}

// The projection with the router rows: W [P, N*C] and W_r [N, N*C] split
// into 64-row stage images (rows 48 .. 48 + N - 1 = W_r), then one pass that
// gives the coefficients (as launch_coeffs_tc) and the router's record
// inputs `zr` [T, P + 1] (rstd W_r v, rstd sum(v), rstd).
cudaError_t launch_coeffs_tc_router(const Params& p, const void* X, const float* W, const float* W_r, void* Wsplit,
                                    float* saved, float* coef, float* zr, cudaStream_t st) {
  using namespace coeffs;
  using L = Layout<true, true>;
  const size_t T_all = (size_t)p.B * p.S;
  const size_t NC = (size_t)p.N * p.C;
  if (p.C % (KC * L::BOXES) != 0 || p.N > L::WR - W_ROWS) return cudaErrorInvalidValue;
  const size_t per_sm = (T_all + sm_count() - 1) / sm_count();
  const int rows = (int)std::min<size_t>(TILE_T, std::max<size_t>(64, (per_sm + 7) / 8 * 8));
  CUtensorMap mx;
  {
    const uint64_t dims[3] = {(uint64_t)p.C, (uint64_t)p.N, T_all};
    const uint64_t strides[2] = {(uint64_t)p.C * 2, NC * 2};
    const uint32_t box[3] = {KC, 1, (uint32_t)rows};
    if (!make_map(&mx, X, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const int ntiles = (int)((T_all + rows - 1) / rows);
  const int grid = std::min(ntiles, sm_count());
  CoeffsOut o{nullptr, nullptr, nullptr, saved, coef, (const uint8_t*)Wsplit, zr};
  const int starve = g_starve_next_projection.exchange(0);
  const size_t threads = (size_t)L::WR * (NC / 8);
  timing_begin("w_split", st);
  w_split_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(W, (uint8_t*)Wsplit, p.P, NC, W_r, p.N, L::WR);
  timing_end(st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaFuncSetAttribute(coeffs_tc_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       smem_bytes<true, true>());
  timing_begin("coeffs_tc_router", st);
  coeffs_tc_kernel<true, true><<<grid, THREADS, smem_bytes<true, true>(), st>>>(mx, mx, mx, p, o, ntiles, rows,
                                                                                starve);
  timing_end(st);
  return cudaGetLastError();
}

// Conv weights w4 [C, 4], w8 [C, 8], w12 [C, 12] -> tap-major per 64-channel
// chunk: taps[cc][r][c'] with rows r = 0..3 the taps of w4, 4..11 those of
// w8, 12..23 those of w12, for channel cc * 64 + c'.
__global__ void taps_major_kernel(const float* __restrict__ w4, const float* __restrict__ w8,
                                  const float* __restrict__ w12, float* __restrict__ taps, int C) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= C * NTAPS) return;
  const int c = i % C, r = i / C;
  const float v = r < 4 ? w4[c * 4 + r] : (r < 12 ? w8[c * 8 + (r - 4)] : w12[c * 12 + (r - 12)]);
  taps[((size_t)(c / flash::KC) * NTAPS + r) * flash::KC + (c % flash::KC)] = v;
}

bool flash_supported(const Params& p) { return p.C % flash::KC == 0 && p.P <= coeffs::W_ROWS && p.k <= KMAX; }
size_t flash_taps_bytes(const Params& p) { return (size_t)NTAPS * p.C * sizeof(float); }

cudaError_t launch_w_split(const Params& p, const float* W, void* Wsplit, cudaStream_t st) {
  const size_t NC = (size_t)p.N * p.C;
  const size_t threads = (size_t)coeffs::W_ROWS * (NC / 8);
  timing_begin("w_split", st);
  w_split_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(W, (uint8_t*)Wsplit, p.P, NC);
  timing_end(st);
  return cudaGetLastError();
}

cudaError_t launch_flash_step(const Params& p, void* X, const void* out, const float* const (&w)[3], float* taps,
                              const float* coef, const void* Wsplit_next, void* x_in, float* coef_next,
                              float* saved_next, cudaStream_t st) {
  using namespace flash;
  const size_t T_all = (size_t)p.B * p.S;
  const bool has_conv = w[0] != nullptr;
  if (has_conv) {
    const int n = p.C * NTAPS;
    timing_begin("taps_major", st);
    taps_major_kernel<<<(n + 255) / 256, 256, 0, st>>>(w[0], w[1], w[2], taps, p.C);
    timing_end(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // tokens per tile as in the coefficient pass: one wave over the SMs where
  // that keeps at least 64 tokens per tile
  const size_t per_sm = (T_all + sm_count() - 1) / sm_count();
  const int rows = (int)std::min<size_t>(TILE_T, std::max<size_t>(64, (per_sm + 7) / 8 * 8));
  CUtensorMap mx, mo;
  {
    const uint64_t dims[3] = {(uint64_t)p.C, (uint64_t)p.N, T_all};
    const uint64_t strides[2] = {(uint64_t)p.C * 2, (uint64_t)p.N * p.C * 2};
    const uint32_t box[3] = {KC, 1, (uint32_t)rows};
    if (!make_map(&mx, X, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)p.C, T_all};
    const uint64_t strides[1] = {(uint64_t)p.C * 2};
    const uint32_t box[2] = {KC, (uint32_t)(rows + HALO_R)};
    if (!make_map(&mo, out, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const int ntiles = (int)((T_all + rows - 1) / rows);
  const int grid = std::min(ntiles, sm_count());
  FlashArgs f{coef, has_conv ? taps : nullptr, (const uint8_t*)Wsplit_next, (__nv_bfloat16*)x_in,
              CoeffsOut{nullptr, nullptr, nullptr, saved_next, coef_next, nullptr}};
  timing_begin("flash_tc", st);
  if (has_conv) {
    cudaFuncSetAttribute(flash_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    flash_tc_kernel<true><<<grid, THREADS, SMEM, st>>>(mx, mo, p, f, ntiles, rows);
  } else {
    cudaFuncSetAttribute(flash_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    flash_tc_kernel<false><<<grid, THREADS, SMEM, st>>>(mx, mo, p, f, ntiles, rows);
  }
  timing_end(st);
  return cudaGetLastError();
}

int read_device_error(cudaStream_t st) {
  int v = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
  }
  return v;
}

// ---------------------------------------------------------------- backward stream pass
//
// dX and dW of every stream on the tensor cores.  Work item = (column block:
// stream n, channels c0 .. c0+127) x (token range); tiles of 128 tokens.
// Per tile, TMA brings
//   Xt   [128 tokens x 128 columns]  the state before the update (two 64-column
//                                     boxes, 128-byte swizzle)
//   Bt   [128 x 128]                 dX' (inactive n) or the active-stream mix
//                                     written to dX by the token pass
//   Pt   [128 tokens x 64]           dp (bf16 hi and lo parts, P <= 48 entries,
//                                     zero padded)
// and the tensor cores compute, with hi + lo parts of dp and of W (about 16
// bits each; the lo x lo product is dropped)
//   dV [128 tokens x 128 cols] = Pt . Wt_blk^T   (A K-major, B K-major; K = 48)
//   dW [128 cols x 48]        += Xt^T . Pt       (A and B MN-major: the same
//                                                 tiles, read along tokens)
// dV goes to a double-buffered TMEM accumulator that the epilogue turns into
// dX = dV + alpha X + base (+ hpre[n] dx_in); dW accumulates in TMEM over the
// whole token range and is written as one partial per range.
//
// The epilogue writes the dX tile into the stage's Pt region (free once both
// contractions have read it), in the same swizzled layout TMA uses, and a
// store warp sends it out with two TMA stores: full 128-byte lines instead of
// one 16-byte piece per token row per store instruction.  The stage's X and B
// part is released as soon as the epilogue has read it, so the next tile's
// HBM loads start while the store is still reading the Pt region; the Pt part
// is released when the store has read it.
//
// Section "Scaling N" (coefficients come from the whole state, so every
// stream receives the projection gradient); section "Dense read, sparse
// write" (inactive streams pass dX' through, active ones receive the mix).

namespace bwdtc {
constexpr int TT = 128;
constexpr int CB = 128;
constexpr int STAGES = 2;
constexpr int HALF = TT * 64 * 2;                 // one 64-column box: 16 KB
constexpr int OFF_X = 0;
constexpr int OFF_B = 2 * HALF;
constexpr int OFF_P = 4 * HALF;                   // dp, hi part; then dX box 0
constexpr int OFF_PL = 5 * HALF;                  // dp, lo part; then dX box 1
constexpr int STAGE_BYTES = 6 * HALF;             // 96 KB
constexpr int WT_BYTES = CB * 64 * 2;             // 16 KB per part of W^T
constexpr int SMEM = STAGES * STAGE_BYTES + 2 * WT_BYTES + 1024;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 32 * (3 + EPI_WARPS);     // producer, MMA issuer, epilogue, store
constexpr int STORE_WARP = 2 + EPI_WARPS;
constexpr int TMEM_COLS = 512;                    // dV: 2 x 128, dW: 48 at column 256
constexpr int D2_COL = 256;
}  // namespace bwdtc

struct StreamMaps {
  CUtensorMap X, Xa, dXp, dX, dP, dPl, Wt, Wtl;
};

// ROUTED: per-token active sets (a.tok_idx) and the router rows of dp / W^T.
template <bool ROUTED>
__global__ void __launch_bounds__(bwdtc::THREADS, 1)
    bwd_stream_tc_kernel(const __grid_constant__ StreamMaps m, Params p, BwdArgs<__nv_bfloat16> a, int ranges,
                         int range_len, float* __restrict__ wpart) {
  using namespace bwdtc;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* wt_s = smem + STAGES * STAGE_BYTES;
  // full: stage loaded; xb_free: X and B read (MMA + epilogue); mma_done: both
  // contractions done with the stage; out_ready: dX tile written to the Pt
  // region; p_free: the store has read it
  __shared__ uint64_t full[STAGES], xb_free[STAGES], mma_done[STAGES], out_ready[STAGES], p_free[STAGES];
  __shared__ uint64_t tfull[2], tempty[2], wt_full, wt_empty, d2full, d2empty, mdrain;
  __shared__ uint32_t tmem_slot;
  int* err = &g_device_error;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, k = p.k, C = p.C, P = p.P;
  const size_t T_all = (size_t)p.B * p.S;
  const size_t NC = (size_t)N * C;
  const int cblocks = C / CB;
  const int nblocks = N * cblocks;
  const int nitems = nblocks * ranges;
  // router: per-token active sets; dp carries N more entries (the W_r rows of
  // W^T), so the contractions run K = 64 (dV) and N = 64 (dW)
  constexpr bool routed = ROUTED;
  const int wrows = routed ? P + N : P;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&xb_free[s], 1 + EPI_WARPS);    // MMA commit + epilogue warps
      mbar_init(&mma_done[s], 1);
      mbar_init(&out_ready[s], EPI_WARPS);
      mbar_init(&p_free[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], EPI_WARPS);
    }
    mbar_init(&wt_full, 1);
    mbar_init(&wt_empty, 1);
    mbar_init(&d2full, 1);
    mbar_init(&d2empty, EPI_WARPS);
    mbar_init(&mdrain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
      int it = 0, ii = 0, issued = 0, nwt = 0;
      for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++ii) {
        const int blk = item / ranges, r = item % ranges;
        const int n = blk / cblocks, c0 = (blk % cblocks) * CB;
        const int slot = p.is_active[n];
        const size_t t_beg = (size_t)r * range_len;
        const size_t t_end = (t_beg + range_len < T_all) ? t_beg + range_len : T_all;
        bool ok = true;
        for (size_t t0 = t_beg; t0 < t_end; t0 += TT, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = ((it / STAGES) & 1) ^ 1;
          if (it >= STAGES && !mbar_wait(&xb_free[s], ph, err, 22)) { ok = false; break; }
          uint8_t* st = smem + s * STAGE_BYTES;
          mbar_expect_tx(&full[s], STAGE_BYTES);
          const int tt = (int)t0;
          for (int h = 0; h < 2; ++h) {
            if (slot && a.saved_active)
              tma_load_3d(st + OFF_X + h * HALF, &m.Xa, &full[s], c0 + 64 * h, slot - 1, tt, pol_stream);
            else
              tma_load_3d(st + OFF_X + h * HALF, &m.X, &full[s], c0 + 64 * h, n, tt, pol_stream);
            if (slot) tma_load_3d(st + OFF_B + h * HALF, &m.dX, &full[s], c0 + 64 * h, n, tt, pol_stream);
            else tma_load_3d(st + OFF_B + h * HALF, &m.dXp, &full[s], c0 + 64 * h, n, tt, pol_stream);
          }
          issued = it + 1;
          if (it >= STAGES && !mbar_wait(&p_free[s], ph, err, 31)) { ok = false; break; }
          tma_load_2d(st + OFF_P, &m.dP, &full[s], 0, tt, pol_keep);
          tma_load_2d(st + OFF_PL, &m.dPl, &full[s], 0, tt, pol_keep);
          if (t0 == t_beg) {
            // this item's W^T block, once the previous item's contractions are done
            if (ii > 0 && !mbar_wait(&wt_empty, (ii - 1) & 1, err, 21)) { ok = false; break; }
            mbar_expect_tx(&wt_full, 2 * WT_BYTES);
            tma_load_2d(wt_s, &m.Wt, &wt_full, 0, (int)((size_t)n * C + c0), pol_keep);
            tma_load_2d(wt_s + WT_BYTES, &m.Wtl, &wt_full, 0, (int)((size_t)n * C + c0), pol_keep);
            ++nwt;
          }
        }
        if (!ok) break;
      }
      // the loads issued land before the CTA may end (a stage whose dp loads
      // were not issued never completes: its wait gives up after the limit,
      // long after its state loads have landed)
      for (int d = issued > STAGES ? issued - STAGES : 0; d < issued; ++d)
        mbar_wait_drain(&full[d % STAGES], (d / STAGES) & 1);
      if (nwt > 0) mbar_wait_drain(&wt_full, (nwt - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_v = idesc_bf16(TT, CB, 0, 0);
      const uint32_t idesc_w = idesc_bf16(CB, routed ? 64 : 48, 1, 1);
      const int ksteps = routed ? 4 : 3;
      const uint32_t wt_addr = smem_u32(wt_s);
      int it = 0, tl = 0, ii = 0;
      for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++ii) {
        const int r = item % ranges;
        const size_t t_beg = (size_t)r * range_len;
        const size_t t_end = (t_beg + range_len < T_all) ? t_beg + range_len : T_all;
        bool ok = true;
        for (size_t t0 = t_beg; t0 < t_end; t0 += TT, ++it, ++tl) {
          const int s = it % STAGES, buf = tl & 1;
          if (!mbar_wait(&full[s], (it / STAGES) & 1, err, 25)) { ok = false; break; }
          if (t0 == t_beg && !mbar_wait(&wt_full, ii & 1, err, 23)) { ok = false; break; }
          if (tl >= 2 && !mbar_wait(&tempty[buf], ((tl >> 1) & 1) ^ 1, err, 26)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
          // dV = dP . Wt^T  (K = 48: three K16 steps inside the 128-byte rows,
          // four with the router rows); hi.hi + hi.lo + lo.hi
#pragma unroll 4
          for (int ks = 0; ks < ksteps; ++ks) {
            const uint64_t ph = sdesc_sw128(st + OFF_P + ks * 32, 16, 1024);
            const uint64_t pl = sdesc_sw128(st + OFF_PL + ks * 32, 16, 1024);
            const uint64_t wh = sdesc_sw128(wt_addr + ks * 32, 16, 1024);
            const uint64_t wl = sdesc_sw128(wt_addr + WT_BYTES + ks * 32, 16, 1024);
            umma_bf16(tmem + buf * 128, ph, wh, idesc_v, ks > 0);
            umma_bf16(tmem + buf * 128, ph, wl, idesc_v, 1);
            umma_bf16(tmem + buf * 128, pl, wh, idesc_v, 1);
          }
          umma_commit(&tfull[buf]);
          // the previous item's dW partial must be drained before this item's
          // first accumulation
          if (t0 == t_beg && ii > 0) {
            if (!mbar_wait(&d2empty, (ii - 1) & 1, err, 24)) { ok = false; break; }
            tc_fence_after();
          }
          // dW += X^T . dP  (K = 128 tokens: eight K16 steps of 16 rows); hi + lo of dp
#pragma unroll
          for (int ks = 0; ks < TT / 16; ++ks) {
            const uint64_t da = sdesc_sw128(st + OFF_X + ks * 2048, HALF, 1024);
            const uint64_t dh = sdesc_sw128(st + OFF_P + ks * 2048, HALF, 1024);
            const uint64_t dl = sdesc_sw128(st + OFF_PL + ks * 2048, HALF, 1024);
            umma_bf16(tmem + D2_COL, da, dh, idesc_w, (t0 == t_beg && ks == 0) ? 0u : 1u);
            umma_bf16(tmem + D2_COL, da, dl, idesc_w, 1);
          }
          umma_commit(&mma_done[s]);
          umma_commit(&xb_free[s]);
        }
        if (!ok) break;
        umma_commit(&d2full);
        umma_commit(&wt_empty);
      }
      umma_commit(&mdrain);
      mbar_wait_drain(&mdrain, 0);
    }
  } else if (warp == STORE_WARP) {
    // ------------------------------------------------ dX tile stores
    if (lane == 0) {
      int it = 0;
      for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
        const int blk = item / ranges, r = item % ranges;
        const int n = blk / cblocks, c0 = (blk % cblocks) * CB;
        const size_t t_beg = (size_t)r * range_len;
        const size_t t_end = (t_beg + range_len < T_all) ? t_beg + range_len : T_all;
        bool ok = true;
        for (size_t t0 = t_beg; t0 < t_end; t0 += TT, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&out_ready[s], (it / STAGES) & 1, err, 30)) { ok = false; break; }
          const uint8_t* st = smem + s * STAGE_BYTES;
          // rows past the last token are clipped by the tensor map
          tma_store_3d(&m.dX, st + OFF_P, c0, n, (int)t0);
          tma_store_3d(&m.dX, st + OFF_PL, c0 + 64, n, (int)t0);
          tma_store_commit();
          tma_store_wait_read0();
          mbar_arrive(&p_free[s]);
        }
        if (!ok) break;
      }
      tma_store_wait0();
    }
  } else {
    // ------------------------------------------------ epilogue: one thread per token / per column
    // warp w reads TMEM lanes 32 (w % 4) .. +31 (its sub-partition); with
    // eight epilogue warps, two share a sub-partition and split the columns
    constexpr int SPLIT = EPI_WARPS / 4, CC = CB / 16 / SPLIT;
    const int q4 = warp & 3, part = (warp - 2) / 4;
    const int row = 32 * q4 + lane;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const int rl = 1 + N + 4 * k;
    int it = 0, tl = 0, ii = 0;
    for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++ii) {
      const int blk = item / ranges, r = item % ranges;
      const int n = blk / cblocks, c0 = (blk % cblocks) * CB;
      const size_t t_beg = (size_t)r * range_len;
      const size_t t_end = (t_beg + range_len < T_all) ? t_beg + range_len : T_all;
      bool ok = true;
      for (size_t t0 = t_beg; t0 < t_end; t0 += TT, ++it, ++tl) {
        const int s = it % STAGES, buf = tl & 1;
        const uint32_t ph = (it / STAGES) & 1;
        const size_t t = t0 + row;
        const bool live = t < T_all;
        float alpha = 0.0f, hp = 0.0f, beta = 0.0f;   // loaded before the waits
        bool act_row = false;                   // router: stream n active for this token
        // router: an active row's base is the mix the column pass wrote to
        // dX; this thread's 64 channels of it, loaded before the waits too
        uint4 mix[ROUTED ? 2 * CC : 1];
        if (live) {
          alpha = a.rec[t * rl];
          if (a.dx_in) hp = a.rec[t * rl + 1 + n];
          if (ROUTED) {
            beta = a.rec[t * rl + 1 + N];
            for (int i = 0; i < k; ++i) act_row |= a.tok_idx[t * k + i] == n;
            if (act_row) {
              const uint4* src = reinterpret_cast<const uint4*>(a.dX + (t * N + n) * (size_t)C + c0 + part * CC * 16);
#pragma unroll
              for (int v = 0; v < 2 * CC; ++v) mix[v] = src[v];
            }
          }
        }
        if (!mbar_wait(&full[s], ph, err, 27)) { ok = false; break; }
        if (!mbar_wait(&tfull[buf], (tl >> 1) & 1, err, 28)) { ok = false; break; }
        if (!mbar_wait(&mma_done[s], ph, err, 32)) { ok = false; break; }
        tc_fence_after();
        uint8_t* st = smem + s * STAGE_BYTES;
#pragma unroll
        for (int ci = 0; ci < CC; ++ci) {
          const int cc = part * CC + ci;
          uint32_t d[16];
          tmem_ld16(tmem + lane_base + buf * 128 + cc * 16, d);
          const int h = cc >> 2;                        // which 64-column box
          const int byte0 = (cc & 3) * 32;              // 16 columns = 32 bytes
          const uint32_t o0 = sw128_offset(row, byte0), o1 = sw128_offset(row, byte0 + 16);
          const uint8_t* xr = st + OFF_X + h * HALF;
          const uint8_t* br = st + OFF_B + h * HALF;
          const uint4 x0 = *reinterpret_cast<const uint4*>(xr + o0);
          const uint4 x1 = *reinterpret_cast<const uint4*>(xr + o1);
          uint4 b0 = *reinterpret_cast<const uint4*>(br + o0);
          uint4 b1 = *reinterpret_cast<const uint4*>(br + o1);
          if (ROUTED && act_row) {
            b0 = mix[2 * ci];
            b1 = mix[2 * ci + 1];
          }
          const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
          float g[16];
          if (a.dx_in && live) {
            float v0[8], v1[8];
            load_vec(a.dx_in + t * C + c0 + cc * 16, v0);
            load_vec(a.dx_in + t * C + c0 + cc * 16 + 8, v1);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              g[e] = v0[e];
              g[8 + e] = v1[e];
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) g[e] = 0.0f;
          }
          tmem_wait_ld();
          uint32_t o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float ya = __uint_as_float(d[2 * e]) + bf_lo(bw[e]);
            float yb = __uint_as_float(d[2 * e + 1]) + bf_hi(bw[e]);
            ya = fmaf(alpha, bf_lo(xw[e]), ya);
            yb = fmaf(alpha, bf_hi(xw[e]), yb);
            ya = fmaf(hp, g[2 * e], ya);
            yb = fmaf(hp, g[2 * e + 1], yb);
            if (ROUTED) {
              ya += beta;
              yb += beta;
            }
            o[e] = pack_bf2(ya, yb);
          }
          uint8_t* orow = st + OFF_P + h * HALF;        // dX box h, same swizzle as the loads
          *reinterpret_cast<uint4*>(orow + o0) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(orow + o1) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        tc_fence_before();
        fence_async_smem();                             // the tile is read by TMA next
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&tempty[buf]);
          mbar_arrive(&xb_free[s]);
          mbar_arrive(&out_ready[s]);
        }
      }
      if (!ok) break;
      // dW partial of this item: TMEM lane = column of the block, 48 columns = q
      if (!mbar_wait(&d2full, ii & 1, err, 29)) break;
      tc_fence_after();
      float* dst = wpart + (size_t)r * wrows * NC + (size_t)n * C + c0 + row;
#pragma unroll 1
      for (int qc = 16 * part; qc < wrows; qc += 16 * SPLIT) {
        uint32_t d[16];
        tmem_ld16(tmem + lane_base + D2_COL + qc, d);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (qc + e < wrows) dst[(size_t)(qc + e) * NC] = __uint_as_float(d[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d2empty);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

int bwd_stream_ranges(const Params& p) {
  const int blocks = p.N * (p.C / bwdtc::CB);
  const size_t tiles = ((size_t)p.B * p.S + bwdtc::TT - 1) / bwdtc::TT;
  if (tiles == 0) return 1;
  // Fewest ranges whose last wave is within 2% of the best wave balance:
  // every range writes a dW partial of P x N x C floats that the reduction
  // reads back.
  const int sms = sm_count();
  double eff_r[17] = {0};
  double best_eff = 0.0;
  for (int r = 1; r <= 16 && (size_t)r <= tiles; ++r) {
    const long items = (long)blocks * r;
    const long waves = (items + sms - 1) / sms;
    eff_r[r] = (double)items / (double)(waves * sms);
    best_eff = std::max(best_eff, eff_r[r]);
  }
  int best = 1;
  while (best < 16 && eff_r[best] < best_eff - 0.02) ++best;
  // no empty range: every range must own at least one tile
  const size_t per = (tiles + best - 1) / best;
  return (int)((tiles + per - 1) / per);
}

cudaError_t launch_bwd_stream_tc(const Params& p, const BwdArgs<__nv_bfloat16>& a, const __nv_bfloat16* Wt,
                                 const __nv_bfloat16* dP, int ranges, float* wpart, cudaStream_t st) {
  using namespace bwdtc;
  const size_t T_all = (size_t)p.B * p.S;
  const size_t NC = (size_t)p.N * p.C;
  StreamMaps m;
  const uint32_t box3[3] = {64, 1, TT};
  {
    const uint64_t dims[3] = {(uint64_t)p.C, (uint64_t)p.N, T_all};
    const uint64_t strides[2] = {(uint64_t)p.C * 2, NC * 2};
    if (!make_map(&m.X, a.X, 3, dims, strides, box3)) return cudaErrorInvalidValue;
    if (!make_map(&m.dXp, a.dXp, 3, dims, strides, box3)) return cudaErrorInvalidValue;
    if (!make_map(&m.dX, a.dX, 3, dims, strides, box3)) return cudaErrorInvalidValue;
  }
  if (a.saved_active) {
    const uint64_t dims[3] = {(uint64_t)p.C, (uint64_t)p.k, T_all};
    const uint64_t strides[2] = {(uint64_t)p.C * 2, (uint64_t)p.k * p.C * 2};
    if (!make_map(&m.Xa, a.saved_active, 3, dims, strides, box3)) return cudaErrorInvalidValue;
  } else {
    m.Xa = m.X;
  }
  {
    const uint64_t dims[2] = {64, T_all};
    const uint64_t strides[1] = {128};
    const uint32_t box[2] = {64, TT};
    if (!make_map(&m.dP, dP, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_map(&m.dPl, dP + T_all * 64, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {64, NC};
    const uint64_t strides[1] = {128};
    const uint32_t box[2] = {64, CB};
    if (!make_map(&m.Wt, Wt, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_map(&m.Wtl, Wt + NC * 64, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const size_t tiles = (T_all + TT - 1) / TT;
  const int range_len = (int)(((tiles + ranges - 1) / ranges) * TT);
  const int nitems = p.N * (p.C / CB) * ranges;
  const int grid = std::min(nitems, sm_count());
  timing_begin("bwd_stream_tc", st);
  if (a.tok_idx) {
    cudaFuncSetAttribute(bwd_stream_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    bwd_stream_tc_kernel<true><<<grid, THREADS, SMEM, st>>>(m, p, a, ranges, range_len, wpart);
  } else {
    cudaFuncSetAttribute(bwd_stream_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    bwd_stream_tc_kernel<false><<<grid, THREADS, SMEM, st>>>(m, p, a, ranges, range_len, wpart);
  }
  timing_end(st);
  return cudaGetLastError();
}

bool tc_bwd_supported(const Params& p) { return p.C % bwdtc::CB == 0 && p.P <= 48; }

}  // namespace xhc
