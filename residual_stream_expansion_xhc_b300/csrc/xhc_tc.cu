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
#include <mutex>

#include "xhc_sm100.cuh"
#include "xhc_tc.cuh"

namespace xhc {

using namespace sm100;

__device__ int g_device_error = 0;

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
//   warps 2..5  split the W tile into bf16 W_hi = bf16(W) and W_lo =
//               bf16(W - W_hi) (swizzled K-major tiles), and, one thread per
//               token, accumulate the sum of squares of each X stage; then the
//               epilogue (rstd, logits, sigmoid, Sinkhorn, stores)
// D[128 x 48] (fp32, TMEM) accumulates X.W_hi^T + X.W_lo^T over all N*C / 64
// stages of a tile, which keeps about 16 mantissa bits of W; two TMEM buffers
// let the epilogue of tile i overlap the MMAs of tile i+1.

namespace coeffs {
constexpr int TILE_T = 128;
constexpr int KC = 64;                  // state entries per stage (128 bytes of bf16)
constexpr int STAGES = 4;
constexpr int X_BYTES = TILE_T * KC * 2;          // 16 KB
constexpr int W_ROWS = 48;                        // padded P
constexpr int WRAW_BYTES = W_ROWS * KC * 4;       // 12 KB fp32 tile from TMA
constexpr int W_BYTES = W_ROWS * KC * 2;          // 6 KB per bf16 part
constexpr int OFF_WRAW = X_BYTES;
constexpr int OFF_WHI = X_BYTES + WRAW_BYTES;
constexpr int OFF_WLO = OFF_WHI + W_BYTES;
constexpr int STAGE_BYTES = OFF_WLO + W_BYTES;    // 40 KB
constexpr int SMEM = STAGES * STAGE_BYTES + 1024;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 128;                    // 2 buffers x 64 columns
}  // namespace coeffs

struct CoeffsOut {
  float* hpre;
  float* hpost;
  float* hres;
  float* saved;
};

__global__ void __launch_bounds__(coeffs::THREADS, 1)
    coeffs_tc_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapW, Params p,
                     CoeffsOut o, int ntiles) {
  using namespace coeffs;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint64_t full[STAGES], bready[STAGES], empty[STAGES], tfull[2], tempty[2];
  __shared__ uint32_t tmem_slot;
  int* err = &g_device_error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cchunks = p.C / KC;
  const int nk = p.N * cchunks;                 // stages per tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);                   // TMA transaction
      mbar_init(&bready[s], 4);                 // W split done by the 4 math warps
      mbar_init(&empty[s], 1);                  // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    fence_mbar_init();
    tma_prefetch_desc(&mapX);
    tma_prefetch_desc(&mapW);
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
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        for (int kc = 0; kc < nk; ++kc, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (it >= STAGES && !mbar_wait(&empty[s], ph ^ 1, err, 11)) goto done_prod;
          uint8_t* st = smem + s * STAGE_BYTES;
          mbar_expect_tx(&full[s], X_BYTES + p.P * KC * 4);
          const int n = kc / cchunks, c0 = (kc % cchunks) * KC;
          tma_load_3d(st, &mapX, &full[s], c0, n, tile * TILE_T, pol_x);
          tma_load_2d_f32(st + OFF_WRAW, &mapW, &full[s], kc * KC, 0, pol_w);
        }
      }
    done_prod:;
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(TILE_T, W_ROWS, 0, 0);
      int it = 0, tl = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tl) {
        const int buf = tl & 1;
        if (tl >= 2 && !mbar_wait(&tempty[buf], ((tl >> 1) & 1) ^ 1, err, 12)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * 64;
        bool ok = true;
        for (int kc = 0; kc < nk; ++kc, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&bready[s], (it / STAGES) & 1, err, 13)) { ok = false; break; }
          tc_fence_after();
          const uint32_t xs = smem_u32(smem + s * STAGE_BYTES);
#pragma unroll
          for (int ks = 0; ks < KC / 16; ++ks) {
            const uint64_t a = sdesc_sw128(xs + ks * 32, 16, 1024);
            const uint64_t bh = sdesc_sw128(xs + OFF_WHI + ks * 32, 16, 1024);
            const uint64_t bl = sdesc_sw128(xs + OFF_WLO + ks * 32, 16, 1024);
            umma_bf16(d, a, bh, idesc, (kc | ks) != 0);
            umma_bf16(d, a, bl, idesc, 1);
          }
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&tfull[buf]);
      }
    }
  } else {
    // ------------------------------------------------ sum of squares + epilogue
    const int row = 32 * (warp & 3) + lane;             // token row == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    int it = 0, tl = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tl) {
      float ss = 0.0f;
      bool ok = true;
      for (int kc = 0; kc < nk; ++kc, ++it) {
        const int s = it % STAGES;
        if (!mbar_wait(&full[s], (it / STAGES) & 1, err, 14)) { ok = false; break; }
        uint8_t* stg = smem + s * STAGE_BYTES;
        // split W: 48 rows x 8 groups of 8 entries, 3 groups per thread
        for (int u = threadIdx.x - 64; u < W_ROWS * 8; u += 128) {
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
        fence_async_smem();
        const uint8_t* xr = stg + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(xr + 16 * c);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float a = bf_lo(w[h]), b = bf_hi(w[h]);
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bready[s]);
      }
      if (!ok) break;
      const int buf = tl & 1;
      if (!mbar_wait(&tfull[buf], (tl >> 1) & 1, err, 15)) break;
      tc_fence_after();
      float pz[W_ROWS];
#pragma unroll
      for (int c = 0; c < W_ROWS; c += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + buf * 64 + c, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) pz[c + j] = __uint_as_float(r[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);

      const size_t t = (size_t)tile * TILE_T + row;
      if (t >= (size_t)p.B * p.S) continue;
      const int N = p.N, k = p.k, P = p.P;
      const float rstd = 1.0f / sqrtf(ss / (float)(N * p.C) + p.eps);
      if (o.saved) {
        float* sv = o.saved + t * (P + 1);
#pragma unroll
        for (int q = 0; q < W_ROWS; ++q)
          if (q < P) sv[q] = rstd * pz[q];
        sv[P] = rstd;
      }
      if (o.hpre) {
#pragma unroll
        for (int q = 0; q < NMAX; ++q)
          if (q < N) o.hpre[t * N + q] = sigmoidf_(rstd * pz[q]);
      }
      if (o.hpost) {
#pragma unroll
        for (int q = 0; q < 4 * KMAX; ++q)
          if (q < 4 * k) o.hpost[t * 4 * k + q] = sigmoidf_(rstd * pz[N + q]);
      }
      if (o.hres) {
        // Sinkhorn of this token's k x k logits in registers (one thread)
        float M[KMAX][KMAX];
        float zmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < KMAX; ++i)
#pragma unroll
          for (int j = 0; j < KMAX; ++j)
            if (i < k && j < k) zmax = fmaxf(zmax, rstd * pz[N + 4 * k + k * i + j]);
#pragma unroll
        for (int i = 0; i < KMAX; ++i)
#pragma unroll
          for (int j = 0; j < KMAX; ++j)
            M[i][j] = (i < k && j < k) ? expf(rstd * pz[N + 4 * k + k * i + j] - zmax) : 0.0f;
        for (int itr = 0; itr < p.iters; ++itr) {
#pragma unroll
          for (int i = 0; i < KMAX; ++i) {
            const float s = (M[i][0] + M[i][1]) + (M[i][2] + M[i][3]);
#pragma unroll
            for (int j = 0; j < KMAX; ++j) M[i][j] = (i < k && j < k) ? M[i][j] / s : 0.0f;
          }
#pragma unroll
          for (int j = 0; j < KMAX; ++j) {
            const float s = (M[0][j] + M[2][j]) + (M[1][j] + M[3][j]);
#pragma unroll
            for (int i = 0; i < KMAX; ++i) M[i][j] = (i < k && j < k) ? M[i][j] / s : 0.0f;
          }
        }
#pragma unroll
        for (int i = 0; i < KMAX; ++i)
#pragma unroll
          for (int j = 0; j < KMAX; ++j)
            if (i < k && j < k) o.hres[t * k * k + k * i + j] = M[i][j];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------- launchers

bool tc_coeffs_supported(const Params& p) { return p.C % coeffs::KC == 0 && p.P <= coeffs::W_ROWS; }

cudaError_t launch_coeffs_tc(const Params& p, const void* X, const float* W, float* hpre, float* hpost,
                             float* hres, float* saved, cudaStream_t st) {
  using namespace coeffs;
  const size_t T_all = (size_t)p.B * p.S;
  const size_t NC = (size_t)p.N * p.C;
  CUtensorMap mx, mw;
  {
    const uint64_t dims[3] = {(uint64_t)p.C, (uint64_t)p.N, T_all};
    const uint64_t strides[2] = {(uint64_t)p.C * 2, NC * 2};
    const uint32_t box[3] = {KC, 1, TILE_T};
    if (!make_map(&mx, X, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {NC, (uint64_t)p.P};
    const uint64_t strides[1] = {NC * 4};
    const uint32_t box[2] = {KC, (uint32_t)p.P};
    if (!make_map(&mw, W, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return cudaErrorInvalidValue;
  }
  const int ntiles = (int)((T_all + TILE_T - 1) / TILE_T);
  const int grid = std::min(ntiles, sm_count());
  cudaFuncSetAttribute(coeffs_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  CoeffsOut o{hpre, hpost, hres, saved};
  timing_begin("coeffs_tc", st);
  coeffs_tc_kernel<<<grid, THREADS, SMEM, st>>>(mx, mw, p, o, ntiles);
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

bool tc_update_supported(const Params&) { return false; }
cudaError_t launch_update_tc(const Params&, const UpdArgs<__nv_bfloat16>&, bool, cudaStream_t) {
  return cudaErrorNotSupported;
}
bool tc_bwd_supported(const Params&) { return false; }
size_t tc_bwd_partial_bytes(const Params&) { return 0; }
cudaError_t launch_bwd_tc(const Params&, const BwdArgs<__nv_bfloat16>&, bool, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace xhc
