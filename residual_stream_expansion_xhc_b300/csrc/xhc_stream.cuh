// Bandwidth-bound CUDA-core passes for bf16 state (see xhc_stream.cu).
#pragma once

#include "xhc_kernels.cuh"

namespace xhc {

// Coefficient block [T, COEF_STRIDE] from saved logits [T, P + 1].
cudaError_t launch_coef(const Params& p, const float* saved, float* coef, cudaStream_t st);

// Forward update from a coefficient block: x_in, saved active rows, sparse write.
bool stream_update_supported(const Params& p);
cudaError_t launch_fwd_update(const Params& p, const UpdArgs<__nv_bfloat16>& a, const float* coef, bool has_conv,
                              int sms, cudaStream_t st);

// Backward column pass: active-stream mix into dX, dout, conv-weight partials
// (rows of [24][C], one per CTA of a channel block) and coefficient dots.
// `taps` is scratch of bwd_col_taps_floats() floats (the tap-major copy of the
// conv weights the pass reads; unused without convolution branches).
size_t bwd_col_pdot_floats(const Params& p);
size_t bwd_col_cpart_floats(const Params& p, int sms);
size_t bwd_col_taps_floats(const Params& p);
int bwd_col_cpart_rows(const Params& p, int sms);
cudaError_t launch_bwd_col(const Params& p, const BwdArgs<__nv_bfloat16>& a, const float* coef, bool has_conv,
                           float* pdot, float* cpart, float* taps, int sms, cudaStream_t st);

// Backward per-token reverse: dp (bf16, 64 per token) and records
// [alpha | hpre (N) | unused (4k)].  With Gram-Schmidt, gsdh [T, 16] holds
// dL/dH^post (from launch_gs_rev) in place of the column pass's dots.
cudaError_t launch_bwd_dz(const Params& p, const float* saved, const float* pdot, bool has_dxin,
                          __nv_bfloat16* dP, float* rec, const float* gsdh, const RouterBwd& rb, cudaStream_t st);

// Gram-Schmidt reverse per token: dL/dH^post [T, 16] into gsdh and the Gram
// term S = dM + dM^T [T, 16] into sgram, from the column pass's dots, the
// saved logits and the per-token T and M records of launch_gs_fold.
cudaError_t launch_gs_rev(const Params& p, const float* saved, const float* pdot, const float* gsrec, float* gsdh,
                          float* sgram, cudaStream_t st);

// Debug builds (XHC_DEBUG): read and clear the first out-of-extent access of
// the streaming kernels (1 and its source line and address; 0: none; -1:
// release build; -2: CUDA error), and run the checker's self-test.
int debug_record(unsigned long long* line, unsigned long long* addr);
int debug_selftest(const float* buf, float* out, cudaStream_t st);

}  // namespace xhc
