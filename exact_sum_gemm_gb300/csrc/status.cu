// Device-side status of the library, and a self-test of its bounded waits.
//
// The tensor-core kernels never wait without a limit: every mbarrier wait
// gives up after a fixed time, the call's outputs become the canonical NaN and
// the kernel sets a bit in a per-device status word (this file).
// det_device_status reads (and optionally clears) that word, so a caller can
// tell a wait that ran out from a NaN input.
//
// det_selftest_wait_timeout launches one small kernel whose bounded wait, the
// same helper the tensor-core kernels use, waits on a barrier that nothing
// ever releases; when the limit passes it records the expiry in the status
// word exactly as they do.  Nothing is copied asynchronously and no memory is
// held, so the kernel simply returns and the context stays usable.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "det_gemm.h"
#include "det_kernels.h"
#include "tc_ptx.cuh"

namespace det {
namespace {

// One word per device that loads the library; zero means no expiry seen.
static __device__ unsigned int g_status_word;

PerDeviceOnce g_status_once;
unsigned* g_status_addr[kMaxDevices] = {};

__global__ void bounded_wait_selftest_kernel(unsigned* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);           // one arrival would complete phase 0; none comes
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !ptx::mbar_wait_ns(&bar, 0, limit_ns)) atomicOr(status, kStatusTimeout);
}

}  // namespace

cudaError_t device_status_word(unsigned** out) {
  cudaError_t e = g_status_once.run([](int dev) {
    void* p = nullptr;
    // in host code the symbol is a host-side stand-in: ask for the device address
    cudaError_t r = cudaGetSymbolAddress(&p, g_status_word);
    if (r == cudaSuccess) g_status_addr[dev] = static_cast<unsigned*>(p);
    return r;
  });
  if (e != cudaSuccess) return e;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  *out = g_status_addr[dev];
  return cudaSuccess;
}

}  // namespace det

extern "C" {

det_status det_device_status(int clear) {
  unsigned* word = nullptr;
  if (det::device_status_word(&word) != cudaSuccess) return DET_ERR_CUDA;
  // every stream of the device (the caller's may be non-blocking) must be done
  if (cudaDeviceSynchronize() != cudaSuccess) return DET_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DET_ERR_CUDA;
  if (clear && v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return DET_ERR_CUDA;
  }
  return (v & det::kStatusTimeout) ? DET_ERR_TIMEOUT : DET_OK;
}

det_status det_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return DET_ERR_INVALID_ARG;
  unsigned* word = nullptr;
  if (det::device_status_word(&word) != cudaSuccess) return DET_ERR_CUDA;
  det::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(word, limit_ns);
  det::note_launch();
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

}  // extern "C"
