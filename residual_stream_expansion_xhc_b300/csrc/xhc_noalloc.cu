// xhc_sublayer_fwd_noalloc: the fused forward for callers that cannot
// allocate device memory.
//
// The fused forward needs scratch: a per-token coefficient block, a bf16 split
// copy of W, and the per-token logits when the caller does not keep them
// (`saved` == NULL).
// Normally the caller hands that scratch in as a workspace.  Some callers have no way to obtain one: code running
// inside a framework's custom-op or plugin hook that may not call the CUDA
// allocator, a process whose memory is owned by a pool it cannot reach from
// this point, or a C caller that only receives its input and output buffers.
// For them this file reserves a fixed scratch area in the library itself, a
// file-scope __device__ array that every GPU which loads the library holds
// until the process exits.  Nothing here calls cudaMalloc or cudaFree.
#include <cuda.h>

#include <mutex>

#include "../../include/xhc.h"

namespace {

// Capacity of the built-in scratch.  At N = 16, k = 4 (P = 48) a bf16 call
// needs 3072 * C bytes for the split copy of W, plus 192 bytes per token with
// `saved` given or 388 without: at C = 2048 about 141,000 tokens fit with
// `saved` and 70,000 without.
constexpr size_t kScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
struct ScratchAddr {
  CUcontext ctx;     // the context the address belongs to
  void* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The host-side
// name g_fwd_scratch is only a stand-in for the symbol, never a device
// address, so the address is looked up with that device current and cached
// per device, together with the context it was found in: a new context on
// the device (after cudaDeviceReset) holds its own copy of the array, which
// is looked up again.  The first lookup in a context makes the driver load
// this module there, which reserves the 32 MiB; it can fail with
// out-of-memory when the device is full.  A failed lookup leaves no error
// behind in the runtime's last-error slot.
// The driver's cuCtxGetCurrent, fetched through the runtime so that the
// library does not link the driver library directly.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CUcontext current_context() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      p = nullptr;
    }
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  CUcontext ctx = nullptr;
  if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

int scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return XHC_ERR_CUDA;
  }
  CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(g_mutex);
  ScratchAddr& c = g_scratch[dev];
  if (!c.ptr || ctx == nullptr || c.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      c.ptr = nullptr;
      return XHC_ERR_CUDA;
    }
    // the runtime makes the primary context current on its first call, so
    // ask again after the lookup
    if (ctx == nullptr) ctx = current_context();
    c.ctx = ctx;
    c.ptr = p;
  }
  *out = c.ptr;
  return XHC_OK;
}

}  // namespace

extern "C" int xhc_sublayer_fwd_noalloc(const xhc_shape_t* sh, const void* X_in, void* X_out, const void* out,
                                        const float* w4, const float* w8, const float* w12, const float* W,
                                        const int32_t* idx, void* x_in, float* saved, void* saved_active,
                                        xhc_stream_t stream) {
  // Sizes are checked before anything touches the GPU.
  const size_t need = xhc_fwd_workspace_need(sh, saved != nullptr);
  if (need > kScratchBytes) return XHC_ERR_WORKSPACE;
  if (need == 0)
    return xhc_sublayer_fwd(sh, X_in, X_out, out, w4, w8, w12, W, idx, x_in, saved, saved_active, nullptr, 0,
                            stream);
  void* scratch = nullptr;
  const int s = scratch_on_current_device(&scratch);
  if (s != XHC_OK) return s;
  // Every coefficient and logit the update reads is written earlier in the
  // same call, so the scratch needs no clearing between calls.
  return xhc_sublayer_fwd(sh, X_in, X_out, out, w4, w8, w12, W, idx, x_in, saved, saved_active, scratch,
                          kScratchBytes, stream);
}
