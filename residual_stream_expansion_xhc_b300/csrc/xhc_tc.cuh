// Tensor-core (tcgen05 / TMEM / TMA) kernels of the xHC update for bf16 state.
#pragma once

#include "xhc_kernels.cuh"

namespace xhc {

bool tc_coeffs_supported(const Params& p);
// Coefficients of every token (any of the outputs may be nullptr; `coef` is
// the [T, COEF_STRIDE] block).  The dense read x_in is not computed here.
// With Wsplit (coeffs_wsplit_bytes() of scratch) W is split into bf16 hi and
// lo parts once, by a small kernel, and the projection streams them; without
// it the projection splits each fp32 W tile on chip.
size_t coeffs_wsplit_bytes(const Params& p);
cudaError_t launch_coeffs_tc(const Params& p, const void* X, const float* W, void* Wsplit, float* hpre,
                             float* hpost, float* hres, float* saved, float* coef, cudaStream_t st);
// Fused stack step (bf16, C % 64 == 0): sublayer l's dense read (x_in,
// nullable), TFA and sparse write of X in place, and the projection of the
// updated state onto W_{l+1} (split by launch_w_split into Wsplit_next) giving
// sublayer l+1's coefficient block and, if saved_next is set, its logits.
// `coef` is sublayer l's block; w = {w4, w8, w12} or all nullptr; `taps`
// (flash_taps_bytes) receives the tap-major copy of the conv weights.
bool flash_supported(const Params& p);
size_t flash_taps_bytes(const Params& p);
cudaError_t launch_w_split(const Params& p, const float* W, void* Wsplit, cudaStream_t st);
cudaError_t launch_flash_step(const Params& p, void* X, const void* out, const float* const (&w)[3], float* taps,
                              const float* coef, const void* Wsplit_next, void* x_in, float* coef_next,
                              float* saved_next, cudaStream_t st);
// Status recorded by bounded device-side waits (0: none); synchronises `st`
// and clears the record.
// The coefficient projection with the router rows W_r carried along (64 MMA
// rows): coefficients as launch_coeffs_tc (saved logits, coefficient block),
// and zr [T, P+1] = (rstd W_r v, rstd sum(v), ..., rstd) for the router.
// Wsplit: coeffs_router_wsplit_bytes() of scratch.
size_t coeffs_router_wsplit_bytes(const Params& p);
cudaError_t launch_coeffs_tc_router(const Params& p, const void* X, const float* W, const float* W_r, void* Wsplit,
                                    float* saved, float* coef, float* zr, cudaStream_t st);
int read_device_error(cudaStream_t st);
// Limit of the bounded device waits for later launches (0: the default 2 s);
// synchronises the device.  0 on success.
int set_wait_limit_ns(unsigned long long ns);
// The next coefficient projection issues no loads (failure-detection test hook).
void starve_next_projection();

// The bf16 backward built from the token pass, the TFA pass, the tensor-core
// stream pass and the reduction (see xhc_bwd.cuh) serves these shapes.
bool tc_bwd_supported(const Params& p);

}  // namespace xhc
