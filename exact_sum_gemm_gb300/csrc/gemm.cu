// Orchestration of one exact GEMM call:
//   1. exponent pre-pass (row maxima and deep-element counts) + tile routing;
//   2. band kernel on the tiles routed to it (narrow exponent spread);
//   3. general Kulisch kernel on the remaining tiles (any exponent spread).
// Both kernels produce the same exact digits, so routing never changes a bit
// of the result (det-train page, "Method": the result does not depend on how
// the computation is split).
//
// Scratch: one stream-ordered allocation per call from a memory pool owned by
// this library (one pool per device, which keeps its memory reserved so that
// repeated calls do not go back to the driver), released on the same stream
// after the kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "det_arith.cuh"
#include "det_gemm_internal.cuh"
#include "det_kernels.h"

namespace det {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pool[kMaxDevices] = {};

cudaError_t device_pool(cudaMemPool_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  if (g_pool[dev] == nullptr) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool;
    e = cudaMemPoolCreate(&pool, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = ~uint64_t(0);
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return e;
    g_pool[dev] = pool;
  }
  *out = g_pool[dev];
  return cudaSuccess;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

size_t scratch_bytes(const GemmArgs& g, int64_t slots) {
  const int64_t tiles = ((g.M + kTile - 1) / kTile) * ((g.N + kTile - 1) / kTile);
  size_t b = align_up(sizeof(int) * size_t(g.M + g.N), 256);        // emax
  b += align_up(sizeof(int) * size_t(g.M + g.N), 256);              // deep
  b += align_up(size_t(tiles), 256);                                 // route
  if (g.P == nullptr) b += sizeof(int64_t) * size_t(slots) * kPlanes * kTile * kTile;
  return b;
}

Scratch carve_scratch(void* base, const GemmArgs& g, int64_t slots) {
  const int64_t tiles = ((g.M + kTile - 1) / kTile) * ((g.N + kTile - 1) / kTile);
  char* p = static_cast<char*>(base);
  Scratch s{};
  s.emaxA = reinterpret_cast<int*>(p);
  s.emaxB = s.emaxA + g.M;
  p += align_up(sizeof(int) * size_t(g.M + g.N), 256);
  s.deepA = reinterpret_cast<int*>(p);
  s.deepB = s.deepA + g.M;
  p += align_up(sizeof(int) * size_t(g.M + g.N), 256);
  s.route = reinterpret_cast<uint8_t*>(p);
  p += align_up(size_t(tiles), 256);
  s.fallback = g.P == nullptr ? reinterpret_cast<int64_t*>(p) : nullptr;
  s.slots = slots;
  return s;
}

cudaError_t run_gemm_with_scratch(const GemmArgs& g, void* scratch, int64_t slots,
                                  cudaStream_t stream) {
  const Scratch s = carve_scratch(scratch, g, slots);
  cudaError_t e = launch_prepass(g, s, stream);
  if (e != cudaSuccess) return e;
  e = launch_band(g, s, stream);
  if (e != cudaSuccess) return e;
  return launch_kulisch(g, s.route, stream);
}

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  const int64_t slots = band_slots(g);
  cudaMemPool_t pool;
  cudaError_t e = device_pool(&pool);
  if (e != cudaSuccess) return e;
  void* scratch = nullptr;
  e = cudaMallocFromPoolAsync(&scratch, scratch_bytes(g, slots), pool, stream);
  if (e != cudaSuccess) return e;
  e = run_gemm_with_scratch(g, scratch, slots, stream);
  cudaError_t f = cudaFreeAsync(scratch, stream);
  return e != cudaSuccess ? e : f;
}

}  // namespace det
