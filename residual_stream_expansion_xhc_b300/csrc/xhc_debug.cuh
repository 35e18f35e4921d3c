// Debug builds (compiled with -DXHC_DEBUG into libxhc_debug.so): the
// bandwidth kernels (forward update, backward column pass, per-token reverse,
// coefficient block) check every global load and store of their big buffers
// against the extents of the buffers their launch was given.  An access that
// lies outside all of them is not performed (a load reads zeros, a store is
// dropped) and the first such access is recorded: the source line of the
// access and its address.  xhc_debug_record() reads and clears the record.
// Nothing traps and the kernel runs on, so a bad index shows up as a record
// (and a parity failure) instead of a fault.  Release builds compile every
// check to `true`.
//
// This header is included by one translation unit (the streaming kernels and
// their launchers), so the device-side tables below exist once.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace xhc {
namespace dbg {

constexpr int kMaxExtents = 24;

struct Extents {
  int n;
  unsigned long long lo[kMaxExtents];
  unsigned long long hi[kMaxExtents];
};

#ifdef XHC_DEBUG
static __constant__ Extents g_ext;
static __device__ unsigned long long g_record[2];   // source line, address

__device__ __forceinline__ bool ok(const void* p, unsigned bytes, int line) {
  const unsigned long long a = (unsigned long long)p;
  for (int i = 0; i < g_ext.n; ++i)
    if (a >= g_ext.lo[i] && a + bytes <= g_ext.hi[i]) return true;
  if (atomicCAS(&g_record[0], 0ull, (unsigned long long)line) == 0ull) g_record[1] = a;
  return false;
}
#else
__device__ __forceinline__ bool ok(const void*, unsigned, int) { return true; }
#endif

// Host side: the buffers of one launch.
struct ExtentList {
  Extents e{};
  ExtentList& add(const void* p, size_t bytes) {
    if (p && bytes && e.n < kMaxExtents) {
      e.lo[e.n] = (unsigned long long)p;
      e.hi[e.n] = (unsigned long long)p + bytes;
      ++e.n;
    }
    return *this;
  }
};

// Make `l` the extents of the next launches on `st` (debug builds; no-op
// otherwise).  The copy is ordered on the stream before those launches.
inline cudaError_t set_extents(const ExtentList& l, cudaStream_t st) {
#ifdef XHC_DEBUG
  return cudaMemcpyToSymbolAsync(g_ext, &l.e, sizeof(Extents), 0, cudaMemcpyHostToDevice, st);
#else
  (void)l;
  (void)st;
  return cudaSuccess;
#endif
}

}  // namespace dbg
}  // namespace xhc
