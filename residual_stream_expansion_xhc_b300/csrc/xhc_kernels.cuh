// Launcher interface between the C ABI (xhc_api.cu) and the kernel files.
#pragma once

#include "xhc_common.cuh"

namespace xhc {

// Optional per-kernel timing (see xhc_timing_enable in the C header): when
// enabled, every launch is bracketed by CUDA events on its stream.
void timing_begin(const char* name, cudaStream_t st);
void timing_end(cudaStream_t st);

template <typename T>
struct UpdArgs {
  const T* X_in;
  T* X_out;              // nullptr: dense read only (x_in), no update
  const T* out;
  const float* w[3];
  const float* hpre;     // [T, N] or nullptr      (used when saved == nullptr)
  const float* hpost;    // [T, k, 4]               (used when saved == nullptr)
  const float* hres;     // [T, k, k]               (used when saved == nullptr)
  const float* saved;    // [T, P+1] (z, rstd): coefficients derived per tile
  T* x_in;               // nullptr: no dense read
  T* saved_active;       // [T, k, C] or nullptr
  int copy_inactive;     // X_out != X_in
  const int32_t* tok_idx = nullptr;   // [T, k] per-token active streams (router), or nullptr: Params::idx
};

// Router side of the per-token reverse (all NULL without a router).
struct RouterBwd {
  const int32_t* tok_idx = nullptr;   // [T, k]
  const float* rrec = nullptr;        // [T, 2N+2]: scores, logits, LN mean, LN sd
  int n_fixed = 0;
  const float* rs = nullptr;          // [N] row sums of W_r
  float* cm = nullptr;                // [T, N] dp_r * LN mean (the dW_r mean term)
};

template <typename T>
struct BwdArgs {
  const T* X;             // state before the update, or after it when saved_active != nullptr
  const T* saved_active;  // [T, k, C] or nullptr
  const T* out;
  const float* w[3];
  const float* W;
  const float* saved;     // [T, P+1]
  const T* dXp;
  const T* dx_in;         // nullptr: no gradient through the dense read
  T* dX;
  T* dout;
  float* dw[3];
  float* dW;
  float* rec;             // per-token records (workspace)
  const int32_t* tok_idx = nullptr;   // [T, k] per-token active streams (router), or nullptr: Params::idx
  const float* rrec = nullptr;        // [T, 2N+2] router record (scores, logits, LN mean, LN sd)
  int n_fixed = 0;                    // router: slots [0, n_fixed) are fixed streams
};

// Active row i of dX' for token t: G_i = dX'[a_i].
template <typename T>
__device__ __forceinline__ const T* grad_row(const Params& p, const BwdArgs<T>& a, size_t t, int i) {
  return a.dXp + (t * p.N + p.idx[i]) * (size_t)p.C;
}

template <typename T>
cudaError_t launch_coeffs_simt(const Params& p, const void* X, const float* W, float* hpre, float* hpost,
                               float* hres, float* saved, void* x_in, cudaStream_t st);
template <typename T>
cudaError_t launch_update_simt(const Params& p, const UpdArgs<T>& a, bool has_conv, cudaStream_t st);
template <typename T>
cudaError_t launch_tfa(const Params& p, const void* out, const float* w4, const float* w8, const float* w12,
                       void* u, cudaStream_t st);
template <typename T>
cudaError_t launch_bwd_simt(const Params& p, const BwdArgs<T>& a, bool has_conv, float* partial, bool do_token,
                            cudaStream_t st);
size_t bwd_tfa_partial_floats(const Params& p);
cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, int sms, cudaStream_t st);

}  // namespace xhc
