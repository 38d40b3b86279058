// det_gemm_partial_noalloc: det_gemm_partial with its working memory in a
// fixed static device array instead of an allocation.
//
// Some callers cannot call cudaMalloc (a plug-in whose host framework owns all
// device memory, or code that must never enter the allocator because it can
// synchronise the device).  For them this entry point runs the same exponent
// pre-pass, band kernel and general kernel as det_gemm_partial, with the
// scratch carved out of g_noalloc_scratch below.  det_gemm_partial keeps the
// fallback digits of the band kernel in its output P, so the scratch holds
// only the per-row exponent maxima, deep counts and the tile routing table.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "det_gemm.h"
#include "det_gemm_internal.cuh"
#include "det_kernels.h"

namespace det {
namespace {

// One array per device that loads the library; kept until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DET_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

// Returns false when the problem needs more scratch than the static array has.
bool noalloc_fits(const GemmArgs& g) {
  return scratch_bytes(g, 0) <= static_cast<size_t>(DET_NOALLOC_SCRATCH_BYTES);
}

cudaError_t launch_gemm_partial_noalloc(const GemmArgs& g, cudaStream_t stream) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return e;
  const int64_t slots = band_slots(g);      // partials keep fallback digits in P itself
  return run_gemm_with_scratch(g, scratch, slots, false, stream);   // no pool slot either
}

}  // namespace det
