// C ABI of the xHC sublayer update: host-side validation and kernel dispatch.
// Declarations and argument conventions: include/xhc.h.
#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/xhc.h"
#include "xhc_kernels.cuh"
#include "xhc_bwd.cuh"
#include "xhc_tc.cuh"
#include "xhc_stream.cuh"
#include "xhc_gs.cuh"
#include "xhc_router.cuh"

using namespace xhc;

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return XHC_OK;
  g_last_cuda_error = (int)e;
  return XHC_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t esize(const xhc_shape_t* sh) { return sh->dtype == XHC_BF16 ? 2 : 4; }

int check_shape(const xhc_shape_t* sh) {
  if (!sh) return XHC_ERR_ARG;
  if (sh->dtype != XHC_F32 && sh->dtype != XHC_BF16) return XHC_ERR_DTYPE;
  if (sh->B < 0 || sh->S < 0 || sh->N < 1 || sh->N > NMAX || sh->C < 1) return XHC_ERR_SHAPE;
  if (sh->k < 1 || sh->k > KMAX || sh->k > sh->N) return XHC_ERR_SHAPE;
  if (sh->sinkhorn_iters < 0 || sh->sinkhorn_iters > ITERS_MAX) return XHC_ERR_SHAPE;
  if (!(sh->eps > 0.0f)) return XHC_ERR_SHAPE;
  if (((size_t)sh->C * esize(sh)) % 16 != 0) return XHC_ERR_ALIGN;
  if ((size_t)sh->B * (size_t)sh->S > (size_t)INT32_MAX) return XHC_ERR_SHAPE;
  if (sh->gram_schmidt != 0 && sh->gram_schmidt != 1) return XHC_ERR_SHAPE;
  return XHC_OK;
}

int check_idx(const xhc_shape_t* sh, const int32_t* idx) {
  if (!idx) return XHC_ERR_INDEX;
  for (int i = 0; i < sh->k; ++i) {
    if (idx[i] < 0 || idx[i] >= sh->N) return XHC_ERR_INDEX;
    for (int j = 0; j < i; ++j)
      if (idx[j] == idx[i]) return XHC_ERR_INDEX;
  }
  return XHC_OK;
}

// Every listed pointer must be non-NULL (when required) and 16-byte aligned.
int check_ptrs(std::initializer_list<const void*> required, std::initializer_list<const void*> optional) {
  for (const void* p : required) {
    if (!p) return XHC_ERR_ARG;
    if (!aligned16(p)) return XHC_ERR_ALIGN;
  }
  for (const void* p : optional)
    if (p && !aligned16(p)) return XHC_ERR_ALIGN;
  return XHC_OK;
}

// conv weights: all three or none
int check_conv(const float* a, const float* b, const float* c, bool* has) {
  const int n = (a != nullptr) + (b != nullptr) + (c != nullptr);
  if (n != 0 && n != 3) return XHC_ERR_ARG;
  *has = n == 3;
  return XHC_OK;
}

Params make_params(const xhc_shape_t* sh, const int32_t* idx) {
  Params p;
  std::memset(&p, 0, sizeof(p));
  p.B = sh->B; p.S = sh->S; p.N = sh->N; p.C = sh->C; p.k = sh->k;
  p.P = sh->N + 4 * sh->k + sh->k * sh->k;
  p.iters = sh->sinkhorn_iters;
  p.eps = sh->eps;
  if (idx) {
    for (int i = 0; i < sh->k; ++i) {
      p.idx[i] = idx[i];
      p.is_active[idx[i]] = i + 1;
    }
    for (int n = 0; n < sh->N; ++n)
      if (!p.is_active[n]) p.inactive[p.n_inactive++] = n;
  }
  return p;
}

size_t round_up(size_t x) { return (x + 255) & ~(size_t)255; }
size_t tokens(const xhc_shape_t* sh) { return (size_t)sh->B * (size_t)sh->S; }

int num_sms() {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  return sms;
}

// Coefficient pass: tensor-core kernel where the shape tiles, else CUDA cores.
// On the tensor-core path the dense read x_in (if requested) is a second,
// bandwidth-bound kernel that takes H^pre from `hpre` or from `saved`.
int run_coeffs(const xhc_shape_t* sh, const Params& p, const void* X, const float* W, float* hpre, float* hpost,
               float* hres, float* saved, void* x_in, cudaStream_t st) {
  if (sh->dtype == XHC_BF16) {
    using T = __nv_bfloat16;
    if (tc_coeffs_supported(p)) {
      int s = cuda_status(launch_coeffs_tc(p, X, W, nullptr, hpre, hpost, hres, saved, nullptr, st));
      if (s || !x_in) return s;
      UpdArgs<T> a{(const T*)X, nullptr, nullptr, {nullptr, nullptr, nullptr}, hpre, nullptr, nullptr,
                   hpre ? nullptr : saved, (T*)x_in, nullptr, 0};
      return cuda_status(launch_update_simt<T>(p, a, false, st));
    }
    return cuda_status(launch_coeffs_simt<T>(p, X, W, hpre, hpost, hres, saved, x_in, st));
  }
  return cuda_status(launch_coeffs_simt<float>(p, X, W, hpre, hpost, hres, saved, x_in, st));
}

// ---------------------------------------------------------------- timing records

struct TimingRec {
  const char* name;
  cudaEvent_t a, b;
};
bool g_timing = false;
std::vector<TimingRec> g_recs;
std::vector<cudaEvent_t> g_pool;
int g_open = -1;
constexpr size_t kMaxRecs = 1 << 16;

cudaEvent_t pooled_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

namespace xhc {
void timing_begin(const char* name, cudaStream_t st) {
  g_open = -1;
  if (!g_timing || g_recs.size() >= kMaxRecs) return;
  TimingRec r{name, pooled_event(), pooled_event()};
  if (!r.a || !r.b) return;
  cudaEventRecord(r.a, st);
  g_recs.push_back(r);
  g_open = (int)g_recs.size() - 1;
}
void timing_end(cudaStream_t st) {
  if (!g_timing || g_open < 0) return;
  cudaEventRecord(g_recs[g_open].b, st);
  g_open = -1;
}
}  // namespace xhc

extern "C" {

int xhc_timing_enable(int on) {
  g_timing = on != 0;
  return XHC_OK;
}

int xhc_timing_collect(char* names, int* counts, float* total_ms, int max_kernels) {
  std::vector<std::string> keys;
  std::vector<int> cnt;
  std::vector<double> tot;
  int status = XHC_OK;
  for (const TimingRec& r : g_recs) {
    float ms = 0.0f;
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.a, r.b);
    if (e != cudaSuccess) status = cuda_status(e);
    size_t i = 0;
    while (i < keys.size() && keys[i] != r.name) ++i;
    if (i == keys.size()) {
      keys.push_back(r.name);
      cnt.push_back(0);
      tot.push_back(0.0);
    }
    cnt[i] += 1;
    tot[i] += ms;
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
  const int n = (int)std::min(keys.size(), (size_t)std::max(max_kernels, 0));
  for (int i = 0; i < n; ++i) {
    if (names) {
      std::strncpy(names + 48 * i, keys[i].c_str(), 47);
      names[48 * i + 47] = 0;
    }
    if (counts) counts[i] = cnt[i];
    if (total_ms) total_ms[i] = (float)tot[i];
  }
  return status == XHC_OK ? n : -status;
}

const char* xhc_status_string(int status) {
  switch (status) {
    case XHC_OK: return "ok";
    case XHC_ERR_SHAPE: return "bad shape";
    case XHC_ERR_INDEX: return "bad active-index list";
    case XHC_ERR_ALIGN: return "pointer or row not 16-byte aligned";
    case XHC_ERR_DTYPE: return "unsupported dtype";
    case XHC_ERR_WORKSPACE: return "workspace missing or too small";
    case XHC_ERR_CUDA: return "CUDA launch failed";
    case XHC_ERR_TIMEOUT: return "bounded device wait timed out";
    case XHC_ERR_ARG: return "required pointer is NULL";
    default: return "unknown status";
  }
}

int xhc_last_cuda_error(void) { return g_last_cuda_error; }

int xhc_device_status(xhc_stream_t stream) {
  const int v = read_device_error((cudaStream_t)stream);
  if (v < 0) return cuda_status(cudaGetLastError());
  return v ? XHC_ERR_TIMEOUT : XHC_OK;
}

int xhc_set_wait_limit_ns(unsigned long long ns) {
  if (set_wait_limit_ns(ns) != 0) return cuda_status(cudaGetLastError());
  return XHC_OK;
}

int xhc_debug_starve_next_projection(void) {
  starve_next_projection();
  return XHC_OK;
}

int xhc_debug_record(unsigned long long* line, unsigned long long* address) {
  return debug_record(line, address);
}

int xhc_debug_selftest(const float* buf, float* out, xhc_stream_t stream) {
  if (!buf || !out || (reinterpret_cast<uintptr_t>(buf) & 15)) return XHC_ERR_ALIGN;
  const int r = debug_selftest(buf, out, (cudaStream_t)stream);
  return r == 0 ? XHC_OK : cuda_status(cudaGetLastError());
}

int xhc_num_logits(const xhc_shape_t* sh) {
  if (!sh) return 0;
  return sh->N + 4 * sh->k + sh->k * sh->k;
}

int xhc_coeffs(const xhc_shape_t* sh, const void* X, const float* W, float* hpre, float* hpost, float* hres,
               float* saved, void* x_in, xhc_stream_t stream) {
  int s = check_shape(sh);
  if (s) return s;
  if (tokens(sh) == 0) return XHC_OK;
  if ((s = check_ptrs({X, W, hpre, hpost, hres}, {saved, x_in}))) return s;
  const Params p = make_params(sh, nullptr);
  return run_coeffs(sh, p, X, W, hpre, hpost, hres, saved, x_in, (cudaStream_t)stream);
}

int xhc_tfa(const xhc_shape_t* sh, const void* out, const float* w4, const float* w8, const float* w12, void* u,
            xhc_stream_t stream) {
  int s = check_shape(sh);
  if (s) return s;
  if (tokens(sh) == 0) return XHC_OK;
  if (sh->gram_schmidt) return XHC_ERR_ARG;          // returns the raw components only
  if ((s = check_ptrs({out, w4, w8, w12, u}, {}))) return s;
  const Params p = make_params(sh, nullptr);
  cudaStream_t st = (cudaStream_t)stream;
  if (sh->dtype == XHC_BF16) return cuda_status(launch_tfa<__nv_bfloat16>(p, out, w4, w8, w12, u, st));
  return cuda_status(launch_tfa<float>(p, out, w4, w8, w12, u, st));
}

int xhc_sparse_update(const xhc_shape_t* sh, const void* X_in, void* X_out, const void* out, const float* w4,
                      const float* w8, const float* w12, const float* hpost, const float* hres, const int32_t* idx,
                      xhc_stream_t stream) {
  int s = check_shape(sh);
  if (s) return s;
  if ((s = check_idx(sh, idx))) return s;
  bool has_conv = false;
  if ((s = check_conv(w4, w8, w12, &has_conv))) return s;
  if (tokens(sh) == 0) return XHC_OK;
  if (sh->gram_schmidt && has_conv) return XHC_ERR_ARG;   // use xhc_sublayer_fwd
  if ((s = check_ptrs({X_in, X_out, out, hpost, hres}, {w4, w8, w12}))) return s;
  const Params p = make_params(sh, idx);
  cudaStream_t st = (cudaStream_t)stream;
  if (sh->dtype == XHC_BF16) {
    using T = __nv_bfloat16;
    UpdArgs<T> a{(const T*)X_in, (T*)X_out, (const T*)out, {w4, w8, w12}, nullptr, hpost, hres, nullptr,
                 nullptr, nullptr, X_out != X_in};
    return cuda_status(launch_update_simt<T>(p, a, has_conv, st));
  }
  UpdArgs<float> a{(const float*)X_in, (float*)X_out, (const float*)out, {w4, w8, w12}, nullptr, hpost, hres,
                   nullptr, nullptr, nullptr, X_out != X_in};
  return cuda_status(launch_update_simt<float>(p, a, has_conv, st));
}

namespace {
// Forward workspace: the coefficient block [T, COEF_STRIDE] and the bf16 hi/lo
// split of W (bf16 tensor-core path), followed by the logits [T, P + 1] when
// the caller keeps none.
bool fwd_uses_coef(const xhc_shape_t* sh, const Params& p) {
  return sh->dtype == XHC_BF16 && tc_coeffs_supported(p) && stream_update_supported(p);
}
size_t fwd_coef_bytes(const xhc_shape_t* sh) { return round_up(tokens(sh) * COEF_STRIDE * sizeof(float)); }
size_t fwd_wsplit_bytes(const xhc_shape_t* sh) {
  const Params p = make_params(sh, nullptr);
  return fwd_uses_coef(sh, p) ? round_up(coeffs_wsplit_bytes(p)) : 0;
}
size_t fwd_z_bytes(const xhc_shape_t* sh) {
  return round_up(tokens(sh) * (size_t)(sh->N + 4 * sh->k + sh->k * sh->k + 1) * sizeof(float));
}
// Gram-Schmidt: per-token Gram partials, one set per 256-channel block
size_t gs_gpart_bytes(const xhc_shape_t* sh) {
  if (!sh->gram_schmidt) return 0;
  const Params p = make_params(sh, nullptr);
  return round_up(tokens(sh) * (size_t)gs_gram_blocks(p) * GS_PSTRIDE * sizeof(float));
}
}  // namespace

size_t xhc_fwd_workspace_bytes(const xhc_shape_t* sh) {
  if (check_shape(sh)) return 0;
  const Params p = make_params(sh, nullptr);
  return (fwd_uses_coef(sh, p) ? fwd_coef_bytes(sh) : 0) + fwd_wsplit_bytes(sh) + fwd_z_bytes(sh) +
         gs_gpart_bytes(sh);
}

size_t xhc_fwd_workspace_need(const xhc_shape_t* sh, int keeps_saved) {
  if (check_shape(sh)) return 0;
  const Params p = make_params(sh, nullptr);
  return (fwd_uses_coef(sh, p) ? fwd_coef_bytes(sh) : 0) + fwd_wsplit_bytes(sh) + (keeps_saved ? 0 : fwd_z_bytes(sh)) +
         gs_gpart_bytes(sh);
}

int xhc_sublayer_fwd(const xhc_shape_t* sh, const void* X_in, void* X_out, const void* out, const float* w4,
                     const float* w8, const float* w12, const float* W, const int32_t* idx, void* x_in, float* saved,
                     void* saved_active, void* workspace, size_t ws_bytes, xhc_stream_t stream) {
  int s = check_shape(sh);
  if (s) return s;
  if ((s = check_idx(sh, idx))) return s;
  bool has_conv = false;
  if ((s = check_conv(w4, w8, w12, &has_conv))) return s;
  if (tokens(sh) == 0) return XHC_OK;
  if ((s = check_ptrs({X_in, X_out, out, W}, {w4, w8, w12, x_in, saved, saved_active, workspace}))) return s;
  const Params p = make_params(sh, idx);
  const bool use_coef = fwd_uses_coef(sh, p);
  const bool gs = sh->gram_schmidt && has_conv;
  if (gs && !use_coef) return XHC_ERR_DTYPE;
  const size_t need = xhc_fwd_workspace_need(sh, saved != nullptr);
  if (need > 0 && (!workspace || ws_bytes < need)) return XHC_ERR_WORKSPACE;
  char* ws = (char*)workspace;
  float* coef = use_coef ? (float*)ws : nullptr;
  void* wsplit = use_coef ? (void*)(ws + fwd_coef_bytes(sh)) : nullptr;
  const size_t z_off = use_coef ? fwd_coef_bytes(sh) + fwd_wsplit_bytes(sh) : 0;
  float* z = saved ? saved : (float*)(ws + z_off);
  float* gpart = gs ? (float*)(ws + z_off + (saved ? 0 : fwd_z_bytes(sh))) : nullptr;
  cudaStream_t st = (cudaStream_t)stream;
  if (use_coef) {
    // coefficients on the tensor cores, then one streaming pass: dense read,
    // TFA and sparse write
    using T = __nv_bfloat16;
    if ((s = cuda_status(launch_coeffs_tc(p, X_in, W, wsplit, nullptr, nullptr, nullptr, z, coef, st)))) return s;
    if (gs) {
      // Gram-Schmidt folded into H^post (section "Conv / Gram-Schmidt")
      const float* const w[3] = {w4, w8, w12};
      if ((s = cuda_status(launch_gs_gram(p, (const T*)out, w, gpart, st)))) return s;
      if ((s = cuda_status(launch_gs_fold(p, gpart, coef, nullptr, st)))) return s;
    }
    UpdArgs<T> a{(const T*)X_in, (T*)X_out, (const T*)out, {w4, w8, w12}, nullptr, nullptr, nullptr, z,
                 (T*)x_in, (T*)saved_active, X_out != X_in};
    return cuda_status(launch_fwd_update(p, a, coef, has_conv, num_sms(), st));
  }
  if ((s = run_coeffs(sh, p, X_in, W, nullptr, nullptr, nullptr, z, x_in, st))) return s;
  if (sh->dtype == XHC_BF16) {
    using T = __nv_bfloat16;
    UpdArgs<T> a{(const T*)X_in, (T*)X_out, (const T*)out, {w4, w8, w12}, nullptr, nullptr, nullptr, z,
                 nullptr, (T*)saved_active, X_out != X_in};
    return cuda_status(launch_update_simt<T>(p, a, has_conv, st));
  }
  UpdArgs<float> a{(const float*)X_in, (float*)X_out, (const float*)out, {w4, w8, w12}, nullptr, nullptr, nullptr,
                   z, nullptr, (float*)saved_active, X_out != X_in};
  return cuda_status(launch_update_simt<float>(p, a, has_conv, st));
}

namespace {
// Router forward workspace: the plain forward's, then the 64-row split of
// [W; W_r] (stage images of the projection that carries the router rows), the
// router's record inputs [T, P+1] and the row sums of W_r.
size_t routed_extra_bytes(const xhc_shape_t* sh) {
  const size_t NC = (size_t)sh->N * sh->C;
  const size_t P = (size_t)(sh->N + 4 * sh->k + sh->k * sh->k);
  return round_up((size_t)2 * 64 * NC * sizeof(uint16_t)) + round_up(tokens(sh) * (P + 1) * sizeof(float)) +
         round_up((size_t)sh->N * sizeof(float));
}

int check_fixed(const xhc_shape_t* sh, const int32_t* fixed, int nf) {
  if (nf < 0 || nf > sh->k || (nf > 0 && !fixed)) return XHC_ERR_INDEX;
  for (int i = 0; i < nf; ++i) {
    if (fixed[i] < 0 || fixed[i] >= sh->N) return XHC_ERR_INDEX;
    for (int j = 0; j < i; ++j)
      if (fixed[j] == fixed[i]) return XHC_ERR_INDEX;
  }
  return XHC_OK;
}
}  // namespace

size_t xhc_fwd_routed_workspace_bytes(const xhc_shape_t* sh) {
  if (check_shape(sh)) return 0;
  return xhc_fwd_workspace_bytes(sh) + routed_extra_bytes(sh);
}

int xhc_sublayer_fwd_routed(const xhc_shape_t* sh, const void* X_in, void* X_out, const void* out, const float* w4,
                            const float* w8, const float* w12, const float* W, const float* W_r,
                            const int32_t* fixed, int n_fixed, void* x_in, float* saved, void* saved_active,
                            int32_t* tok_idx, float* rrec, void* workspace, size_t ws_bytes,
                            xhc_stream_t stream) {
  int s = check_shape(sh);
  if (s) return s;
  if (sh->gram_schmidt) return XHC_ERR_ARG;           // not combined with the router
  if ((s = check_fixed(sh, fixed, n_fixed))) return s;
  bool has_conv = false;
  if ((s = check_conv(w4, w8, w12, &has_conv))) return s;
  if (tokens(sh) == 0) return XHC_OK;
  if ((s = check_ptrs({X_in, X_out, out, W, W_r, tok_idx, rrec, workspace},
                      {w4, w8, w12, x_in, saved, saved_active})))
    return s;
  const Params p = make_params(sh, nullptr);
  if (!fwd_uses_coef(sh, p)) return XHC_ERR_DTYPE;     // bf16 tensor-core path only
  if (ws_bytes < xhc_fwd_routed_workspace_bytes(sh)) return XHC_ERR_WORKSPACE;
  char* ws = (char*)workspace;
  float* coef = (float*)ws;
  void* wsplit = ws + fwd_coef_bytes(sh);
  float* zw = (float*)(ws + fwd_coef_bytes(sh) + fwd_wsplit_bytes(sh));
  float* z = saved ? saved : zw;
  (void)wsplit;                                        // the router's projection uses its own 64-row split
  char* rbase = ws + xhc_fwd_workspace_bytes(sh);
  const size_t NC = (size_t)p.N * p.C;
  void* wsplit_r = rbase;
  float* zr = (float*)(rbase + round_up((size_t)2 * 64 * NC * sizeof(uint16_t)));
  float* rs = (float*)((char*)zr + round_up(tokens(sh) * (size_t)(p.P + 1) * sizeof(float)));
  cudaStream_t st = (cudaStream_t)stream;
  using T = __nv_bfloat16;
  // one projection pass gives the coefficients and the router's logits
  // (W_r rides along as 16 more MMA rows); then the routing
  if ((s = cuda_status(launch_router_rowsums(p, W_r, rs, st)))) return s;
  if ((s = cuda_status(launch_coeffs_tc_router(p, X_in, W, W_r, wsplit_r, z, coef, zr, st)))) return s;
  if ((s = cuda_status(launch_route(p, zr, rs, fixed, n_fixed, tok_idx, rrec, coef, st)))) return s;
  UpdArgs<T> a{(const T*)X_in, (T*)X_out, (const T*)out, {w4, w8, w12}, nullptr, nullptr, nullptr, z,
               (T*)x_in, (T*)saved_active, X_out != X_in, tok_idx};
  return cuda_status(launch_fwd_update(p, a, coef, has_conv, num_sms(), st));
}

namespace {
// Workspace of the backward.  CUDA-core path: per-token records (2P+1 floats),
// recomputed logits, conv partials.  bf16 tensor-core path: records
// (1+N+4k floats), recomputed logits, dp (bf16 hi and lo parts, 64 each per
// token), W^T (bf16 hi and lo parts, 64 each per column), the coefficient block, the column pass's coefficient dots and
// conv partials, dW partials (one per token range).
struct BwdLayout {
  size_t rec, saved, dP, Wt, coef, pdot, cpart, wpart, wsplit, gpart, gsrec, sgram, gsdh, ctaps, total;
  int ranges, cpart_rows, col_rows;
};
BwdLayout bwd_layout(const xhc_shape_t* sh) {
  const Params p = make_params(sh, nullptr);
  const size_t T = tokens(sh);
  const size_t NC = (size_t)p.N * p.C;
  BwdLayout L{};
  if (sh->dtype == XHC_BF16 && tc_bwd_supported(p)) {
    const int sms = num_sms();
    L.ranges = bwd_stream_ranges(p);
    L.col_rows = bwd_col_cpart_rows(p, sms);
    // Gram-Schmidt adds one conv-weight partial row per token range of its pass
    L.cpart_rows = L.col_rows + (sh->gram_schmidt ? gs_bwd_rows(p) : 0);
    L.rec = 0;
    L.saved = L.rec + round_up(T * (size_t)(1 + p.N + 4 * p.k) * sizeof(float));
    L.dP = L.saved + round_up(T * (size_t)(p.P + 1) * sizeof(float));
    L.Wt = L.dP + round_up(2 * T * 64 * sizeof(uint16_t));
    L.coef = L.Wt + round_up(2 * NC * 64 * sizeof(uint16_t));
    L.pdot = L.coef + round_up(T * COEF_STRIDE * sizeof(float));
    L.cpart = L.pdot + round_up(bwd_col_pdot_floats(p) * sizeof(float));
    L.wpart = L.cpart + round_up((size_t)L.cpart_rows * NTAPS * p.C * sizeof(float));
    L.wsplit = L.wpart + round_up((size_t)L.ranges * p.P * NC * sizeof(float));
    L.gpart = L.wsplit + (tc_coeffs_supported(p) ? round_up(coeffs_wsplit_bytes(p)) : 0);
    L.gsrec = L.gpart + gs_gpart_bytes(sh);
    L.sgram = L.gsrec + (sh->gram_schmidt ? round_up(T * GS_REC * sizeof(float)) : 0);
    L.gsdh = L.sgram + (sh->gram_schmidt ? round_up(T * 16 * sizeof(float)) : 0);
    L.ctaps = L.gsdh + (sh->gram_schmidt ? round_up(T * 16 * sizeof(float)) : 0);
    L.total = L.ctaps + round_up(bwd_col_taps_floats(p) * sizeof(float));
  } else {
    L.rec = 0;
    L.saved = round_up(T * (size_t)(2 * p.P + 1) * sizeof(float));
    L.cpart = L.saved + round_up(T * (size_t)(p.P + 1) * sizeof(float));
    L.total = L.cpart + round_up(bwd_tfa_partial_floats(p) * sizeof(float));
  }
  return L;
}
}  // namespace

// ---------------------------------------------------------------- fused stack forward

namespace {
// Stack workspace: two coefficient blocks (sublayer l read, l+1 written), the
// bf16 split of the next W, the tap-major conv weights, Gram partials.
size_t stack_taps_bytes(const xhc_shape_t* sh) {
  return round_up((size_t)NTAPS * (size_t)sh->C * sizeof(float));
}
size_t stack_wsplit_bytes(const xhc_shape_t* sh) {
  return round_up(coeffs_wsplit_bytes(make_params(sh, nullptr)));
}
}  // namespace

size_t xhc_stack_fwd_workspace_bytes(const xhc_shape_t* sh) {
  if (check_shape(sh)) return 0;
  return 2 * fwd_coef_bytes(sh) + stack_wsplit_bytes(sh) + stack_taps_bytes(sh) + gs_gpart_bytes(sh);
}

int xhc_stack_fwd(const xhc_shape_t* sh, int L, void* X, const void* const* out, const float* const* w4,
                  const float* const* w8, const float* const* w12, const float* const* W, const int32_t* idx,
                  void* const* x_in, float* const* saved, void* workspace, size_t ws_bytes, xhc_stream_t stream) {
  int s = check_shape(sh);
  if (s) return s;
  if (L < 1 || !out || !W || !idx) return XHC_ERR_ARG;
  if (sh->dtype != XHC_BF16) return XHC_ERR_DTYPE;
  const Params p0 = make_params(sh, nullptr);
  if (!flash_supported(p0) || !tc_coeffs_supported(p0) || !stream_update_supported(p0)) return XHC_ERR_SHAPE;
  const int nconv = (w4 != nullptr) + (w8 != nullptr) + (w12 != nullptr);
  if (nconv != 0 && nconv != 3) return XHC_ERR_ARG;
  std::vector<bool> conv(L, false);
  for (int l = 0; l < L; ++l) {
    if ((s = check_idx(sh, idx + (size_t)l * sh->k))) return s;
    bool has = false;
    if (nconv && (s = check_conv(w4[l], w8[l], w12[l], &has))) return s;
    conv[l] = has;
    if ((s = check_ptrs({out[l], W[l]}, {nconv ? w4[l] : nullptr, nconv ? w8[l] : nullptr,
                                         nconv ? w12[l] : nullptr, x_in ? x_in[l] : nullptr,
                                         saved ? saved[l] : nullptr})))
      return s;
  }
  if ((s = check_ptrs({X}, {workspace}))) return s;
  if (tokens(sh) == 0) return XHC_OK;
  const size_t need = xhc_stack_fwd_workspace_bytes(sh);
  if (!workspace || ws_bytes < need) return XHC_ERR_WORKSPACE;
  char* ws = (char*)workspace;
  float* coef[2] = {(float*)ws, (float*)(ws + fwd_coef_bytes(sh))};
  void* wsplit = ws + 2 * fwd_coef_bytes(sh);
  float* taps = (float*)(ws + 2 * fwd_coef_bytes(sh) + stack_wsplit_bytes(sh));
  float* gpart = (float*)(ws + 2 * fwd_coef_bytes(sh) + stack_wsplit_bytes(sh) + stack_taps_bytes(sh));
  cudaStream_t st = (cudaStream_t)stream;
  using T = __nv_bfloat16;
  auto weights = [&](int l, const float* (&w)[3]) {
    w[0] = conv[l] ? w4[l] : nullptr;
    w[1] = conv[l] ? w8[l] : nullptr;
    w[2] = conv[l] ? w12[l] : nullptr;
  };
  // Gram-Schmidt of sublayer l's components folded into its coefficient block
  auto fold = [&](const Params& p, int l, float* cf) -> int {
    if (!sh->gram_schmidt || !conv[l]) return XHC_OK;
    const float* w[3];
    weights(l, w);
    const float* const wc[3] = {w[0], w[1], w[2]};
    int r = cuda_status(launch_gs_gram(p, (const T*)out[l], wc, gpart, st));
    return r ? r : cuda_status(launch_gs_fold(p, gpart, cf, nullptr, st));
  };
  Params p = make_params(sh, idx);
  if ((s = cuda_status(launch_coeffs_tc(p, X, W[0], wsplit, nullptr, nullptr, nullptr, saved ? saved[0] : nullptr,
                                        coef[0], st))))
    return s;
  if ((s = fold(p, 0, coef[0]))) return s;
  for (int l = 0; l < L; ++l) {
    p = make_params(sh, idx + (size_t)l * sh->k);
    const float* w[3];
    weights(l, w);
    float* cur = coef[l & 1];
    float* nxt = coef[(l + 1) & 1];
    if (l + 1 < L) {
      if ((s = cuda_status(launch_w_split(p, W[l + 1], wsplit, st)))) return s;
      const float* const wc[3] = {w[0], w[1], w[2]};
      if ((s = cuda_status(launch_flash_step(p, X, out[l], wc, taps, cur, wsplit, x_in ? x_in[l] : nullptr, nxt,
                                             saved ? saved[l + 1] : nullptr, st))))
        return s;
      if ((s = fold(make_params(sh, idx + (size_t)(l + 1) * sh->k), l + 1, nxt))) return s;
    } else {
      UpdArgs<T> a{(const T*)X, (T*)X, (const T*)out[l], {w[0], w[1], w[2]}, nullptr, nullptr, nullptr, nullptr,
                   x_in ? (T*)x_in[l] : nullptr, nullptr, 0};
      if ((s = cuda_status(launch_fwd_update(p, a, cur, conv[l], num_sms(), st)))) return s;
    }
  }
  return XHC_OK;
}

size_t xhc_bwd_workspace_bytes(const xhc_shape_t* sh) {
  if (check_shape(sh)) return 0;
  return bwd_layout(sh).total;
}

int xhc_sublayer_bwd(const xhc_shape_t* sh, const void* X_state, const void* saved_active, const void* out,
                     const float* w4, const float* w8, const float* w12, const float* W, const int32_t* idx,
                     const float* saved, const void* dXp, const void* dx_in, void* dX, void* dout, float* dw4,
                     float* dw8, float* dw12, float* dW, void* workspace, size_t ws_bytes, xhc_stream_t stream) {
  int s = check_shape(sh);
  if (s) return s;
  if ((s = check_idx(sh, idx))) return s;
  bool has_conv = false;
  if ((s = check_conv(w4, w8, w12, &has_conv))) return s;
  bool has_dconv = false;
  if ((s = check_conv(dw4, dw8, dw12, &has_dconv))) return s;
  if (has_conv != has_dconv) return XHC_ERR_ARG;
  if (saved_active && !saved) return XHC_ERR_ARG;   // recomputation needs the pre-update state
  if (dX == dXp) return XHC_ERR_ARG;                // dX must not alias dX'
  if ((s = check_ptrs({X_state, out, W, dXp, dX, dout, dW}, {saved_active, w4, w8, w12, saved, dx_in, dw4, dw8,
                                                              dw12, workspace})))
    return s;
  const BwdLayout L = bwd_layout(sh);
  if (tokens(sh) == 0) {
    // empty batch: weight gradients are sums over no tokens
    cudaStream_t st = (cudaStream_t)stream;
    const Params p = make_params(sh, idx);
    cudaError_t e = cudaMemsetAsync(dW, 0, (size_t)p.P * p.N * p.C * sizeof(float), st);
    if (has_conv && e == cudaSuccess) e = cudaMemsetAsync(dw4, 0, (size_t)p.C * 4 * sizeof(float), st);
    if (has_conv && e == cudaSuccess) e = cudaMemsetAsync(dw8, 0, (size_t)p.C * 8 * sizeof(float), st);
    if (has_conv && e == cudaSuccess) e = cudaMemsetAsync(dw12, 0, (size_t)p.C * 12 * sizeof(float), st);
    return cuda_status(e);
  }
  if (!workspace || ws_bytes < L.total) return XHC_ERR_WORKSPACE;
  char* ws = (char*)workspace;
  const Params p = make_params(sh, idx);
  cudaStream_t st = (cudaStream_t)stream;
  float* rec = (float*)(ws + L.rec);
  const bool tc_path = sh->dtype == XHC_BF16 && tc_bwd_supported(p);
  const bool gs = sh->gram_schmidt && has_conv;
  if (gs && !tc_path) return XHC_ERR_DTYPE;
  float* coef = tc_path ? (float*)(ws + L.coef) : nullptr;
  bool have_coef = false;
  const float* z = saved;
  if (!z) {
    float* zw = (float*)(ws + L.saved);
    if (tc_path && tc_coeffs_supported(p)) {
      if ((s = cuda_status(launch_coeffs_tc(p, X_state, W, ws + L.wsplit, nullptr, nullptr, nullptr, zw, coef, st))))
        return s;
      have_coef = true;
    } else if ((s = run_coeffs(sh, p, X_state, W, nullptr, nullptr, nullptr, zw, nullptr, st))) {
      return s;
    }
    z = zw;
  }
  if (sh->dtype == XHC_BF16) {
    using T = __nv_bfloat16;
    BwdArgs<T> a{(const T*)X_state, (const T*)saved_active, (const T*)out, {w4, w8, w12}, W, z, (const T*)dXp,
                 (const T*)dx_in, (T*)dX, (T*)dout, {dw4, dw8, dw12}, dW, rec};
    if (tc_path) {
      T* dP = (T*)(ws + L.dP);
      T* Wt = (T*)(ws + L.Wt);
      float* pdot = (float*)(ws + L.pdot);
      float* cpart = (float*)(ws + L.cpart);
      float* wpart = (float*)(ws + L.wpart);
      const int sms = num_sms();
      float* gsrec = gs ? (float*)(ws + L.gsrec) : nullptr;
      float* sgram = gs ? (float*)(ws + L.sgram) : nullptr;
      float* gsdh = gs ? (float*)(ws + L.gsdh) : nullptr;
      const float* const w[3] = {w4, w8, w12};
      if (have_coef) {
        if ((s = cuda_status(launch_wt_prep(p, W, Wt, st)))) return s;
      } else if ((s = cuda_status(launch_bwd_prep(p, W, nullptr, Wt, z, coef, st)))) {
        return s;
      }
      if (gs) {
        // the forward's Gram-Schmidt coefficients again: H^post' in the block, T and M per token
        if ((s = cuda_status(launch_gs_gram(p, (const T*)out, w, (float*)(ws + L.gpart), st)))) return s;
        if ((s = cuda_status(launch_gs_fold(p, (const float*)(ws + L.gpart), coef, gsrec, st)))) return s;
      }
      if ((s = cuda_status(launch_bwd_col(p, a, coef, has_conv, pdot, cpart, (float*)(ws + L.ctaps), sms, st))))
        return s;
      if (gs && (s = cuda_status(launch_gs_rev(p, z, pdot, gsrec, gsdh, sgram, st)))) return s;
      if ((s = cuda_status(launch_bwd_dz(p, z, pdot, dx_in != nullptr, dP, rec, gsdh, RouterBwd{}, st)))) return s;
      if (gs && (s = cuda_status(launch_gs_bwd(p, (const T*)out, w, sgram, (T*)dout,
                                               cpart + (size_t)L.col_rows * NTAPS * p.C, st))))
        return s;
      if ((s = cuda_status(launch_bwd_stream_tc(p, a, Wt, dP, L.ranges, wpart, st)))) return s;
      return cuda_status(launch_bwd_reduce(p, a, has_conv, cpart, L.cpart_rows, L.ranges, wpart, st));
    }
    return cuda_status(launch_bwd_simt<T>(p, a, has_conv, (float*)(ws + L.cpart), true, st));
  }
  BwdArgs<float> a{(const float*)X_state, (const float*)saved_active, (const float*)out, {w4, w8, w12}, W, z,
                   (const float*)dXp, (const float*)dx_in, (float*)dX, (float*)dout, {dw4, dw8, dw12}, dW, rec};
  return cuda_status(launch_bwd_simt<float>(p, a, has_conv, (float*)(ws + L.cpart), true, st));
}

int xhc_hres_active_weights(const xhc_shape_t* sh, const float* W_pp, const float* W_ra, const int32_t* idx,
                            float* W, xhc_stream_t stream) {
  int s = check_shape(sh);
  if (s) return s;
  if ((s = check_idx(sh, idx))) return s;
  if (sh->C % 4) return XHC_ERR_ALIGN;
  if ((s = check_ptrs({W_pp, W_ra, W}, {}))) return s;
  return cuda_status(launch_hres_active_weights(make_params(sh, idx), W_pp, W_ra, W, (cudaStream_t)stream));
}

int xhc_hres_active_grad(const xhc_shape_t* sh, const float* dW, const int32_t* idx, float* dW_ra,
                         xhc_stream_t stream) {
  int s = check_shape(sh);
  if (s) return s;
  if ((s = check_idx(sh, idx))) return s;
  if (sh->C % 4) return XHC_ERR_ALIGN;
  if ((s = check_ptrs({dW, dW_ra}, {}))) return s;
  return cuda_status(launch_hres_active_grad(make_params(sh, idx), dW, dW_ra, (cudaStream_t)stream));
}

namespace {
// Router backward workspace: the plain backward's layout with P + N rows per
// dW partial, then cm [T, N], c_r [N] and rs [N].
struct RoutedBwdLayout {
  BwdLayout L;
  size_t wpart, cm, cr, rs, total;
};
RoutedBwdLayout routed_bwd_layout(const xhc_shape_t* sh) {
  RoutedBwdLayout R{};
  R.L = bwd_layout(sh);
  const Params p = make_params(sh, nullptr);
  const size_t NC = (size_t)p.N * p.C;
  R.wpart = R.L.total;
  R.cm = R.wpart + round_up((size_t)R.L.ranges * (p.P + p.N) * NC * sizeof(float));
  R.cr = R.cm + round_up(tokens(sh) * p.N * sizeof(float));
  R.rs = R.cr + round_up((size_t)p.N * sizeof(float));
  R.total = R.rs + round_up((size_t)p.N * sizeof(float));
  return R;
}
}  // namespace

size_t xhc_bwd_routed_workspace_bytes(const xhc_shape_t* sh) {
  if (check_shape(sh)) return 0;
  return routed_bwd_layout(sh).total;
}

int xhc_sublayer_bwd_routed(const xhc_shape_t* sh, void* X_state, const void* saved_active, const void* out, const float* w4,
                            const float* w8, const float* w12, const float* W, const float* W_r,
                            const int32_t* fixed, int n_fixed, const float* saved, const int32_t* tok_idx,
                            const float* rrec, const void* dXp, const void* dx_in, void* dX, void* dout,
                            float* dw4, float* dw8, float* dw12, float* dW, float* dW_r, void* workspace,
                            size_t ws_bytes, xhc_stream_t stream) {
  int s = check_shape(sh);
  if (s) return s;
  if (sh->gram_schmidt) return XHC_ERR_ARG;
  if ((s = check_fixed(sh, fixed, n_fixed))) return s;
  bool has_conv = false, has_dconv = false;
  if ((s = check_conv(w4, w8, w12, &has_conv))) return s;
  if ((s = check_conv(dw4, dw8, dw12, &has_dconv))) return s;
  if (has_conv != has_dconv) return XHC_ERR_ARG;
  if (dX == dXp) return XHC_ERR_ARG;
  if ((s = check_ptrs({X_state, out, W, W_r, saved, tok_idx, rrec, dXp, dX, dout, dW, dW_r, workspace},
                      {w4, w8, w12, dx_in, dw4, dw8, dw12, saved_active})))
    return s;
  const Params p = make_params(sh, nullptr);
  if (!(sh->dtype == XHC_BF16 && tc_bwd_supported(p)) || p.P + p.N > 64) return XHC_ERR_DTYPE;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t NC = (size_t)p.N * p.C;
  if (tokens(sh) == 0) {
    cudaError_t e = cudaMemsetAsync(dW, 0, (size_t)p.P * NC * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dW_r, 0, (size_t)p.N * NC * sizeof(float), st);
    if (has_conv && e == cudaSuccess) e = cudaMemsetAsync(dw4, 0, (size_t)p.C * 4 * sizeof(float), st);
    if (has_conv && e == cudaSuccess) e = cudaMemsetAsync(dw8, 0, (size_t)p.C * 8 * sizeof(float), st);
    if (has_conv && e == cudaSuccess) e = cudaMemsetAsync(dw12, 0, (size_t)p.C * 12 * sizeof(float), st);
    return cuda_status(e);
  }
  const RoutedBwdLayout R = routed_bwd_layout(sh);
  if (ws_bytes < R.total) return XHC_ERR_WORKSPACE;
  char* ws = (char*)workspace;
  const BwdLayout& L = R.L;
  using T = __nv_bfloat16;
  float* coef = (float*)(ws + L.coef);
  T* dP = (T*)(ws + L.dP);
  T* Wt = (T*)(ws + L.Wt);
  float* pdot = (float*)(ws + L.pdot);
  float* cpart = (float*)(ws + L.cpart);
  float* wpart = (float*)(ws + R.wpart);
  float* cm = (float*)(ws + R.cm);
  float* cr = (float*)(ws + R.cr);
  float* rs = (float*)(ws + R.rs);
  BwdArgs<T> a{(const T*)X_state, nullptr, (const T*)out, {w4, w8, w12}, W, saved, (const T*)dXp, (const T*)dx_in,
               (T*)dX, (T*)dout, {dw4, dw8, dw12}, dW, (float*)(ws + L.rec)};
  a.tok_idx = tok_idx;
  a.rrec = rrec;
  a.n_fixed = n_fixed;
  RouterBwd rb;
  rb.tok_idx = tok_idx;
  rb.rrec = rrec;
  rb.n_fixed = n_fixed;
  rb.rs = rs;
  rb.cm = cm;
  const int sms = num_sms();
  // after an in-place forward: the state before the update first
  if (saved_active && (s = cuda_status(launch_restore_active(p, X_state, saved_active, tok_idx, sms, st)))) return s;
  if ((s = cuda_status(launch_bwd_prep(p, W, W_r, Wt, saved, coef, st)))) return s;
  if ((s = cuda_status(launch_route_scale(p, tok_idx, rrec, n_fixed, coef, st)))) return s;
  if ((s = cuda_status(launch_router_rowsums(p, W_r, rs, st)))) return s;
  if ((s = cuda_status(launch_bwd_col(p, a, coef, has_conv, pdot, cpart, (float*)(ws + L.ctaps), sms, st))))
    return s;
  if ((s = cuda_status(launch_bwd_dz(p, saved, pdot, dx_in != nullptr, dP, a.rec, nullptr, rb, st)))) return s;
  if ((s = cuda_status(launch_bwd_stream_tc(p, a, Wt, dP, L.ranges, wpart, st)))) return s;
  return cuda_status(launch_bwd_reduce(p, a, has_conv, cpart, L.cpart_rows, L.ranges, wpart, st, dW_r, cm, cr));
}

int xhc_copy(const void* src, void* dst, size_t bytes, xhc_stream_t stream) {
  if (!src || !dst) return XHC_ERR_ARG;
  if (!aligned16(src) || !aligned16(dst) || bytes % 16) return XHC_ERR_ALIGN;
  if (bytes == 0) return XHC_OK;
  return cuda_status(launch_copy16(src, dst, bytes, num_sms(), (cudaStream_t)stream));
}

}  // extern "C"
