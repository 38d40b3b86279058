// Orchestration of one exact GEMM call:
//   1. exponent pre-pass (row maxima and deep-element counts) + tile routing;
//   2. residue path on the tiles with few deep elements: bf16 residue planes,
//      residue GEMM on tcgen05 tensor cores, CRT reconstruction + deep
//      products, round once (or digits out);
//   3. general Kulisch kernel on the remaining tiles (any exponent spread).
// With K = 0 (or a grid beyond the tensor-core kernel's limits) the band
// kernel takes the place of step 2.  Every path produces the same exact
// digits, so routing never changes a bit of the result (det-train page,
// "Method": the result does not depend on how the computation is split).
//
// Scratch: one stream-ordered allocation per call from a memory pool owned by
// this library (one pool per device, which keeps its memory reserved so that
// repeated calls do not go back to the driver), released on the same stream
// after the kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include <math.h>

#include <atomic>
#include <mutex>

#include "det_arith.cuh"
#include "det_gemm_internal.cuh"
#include "det_kernels.h"
#include "det_residue.cuh"

namespace det {
namespace {

std::mutex g_pool_mu;
cudaMemPool_t g_pool[kMaxDevices] = {};
uint64_t g_retention = ~uint64_t(0);          // release threshold of the pools (bytes kept)
std::atomic<uint64_t> g_pool_allocs{0};       // allocations taken from the pools

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
    uint64_t keep = g_retention;
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return e;
    g_pool[dev] = pool;
  }
  *out = g_pool[dev];
  return cudaSuccess;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

ResidueOperand residue_operand(const void* X, int64_t ld, int op, int64_t rows, int64_t K, int64_t Kp,
                               int* emax, __nv_bfloat16* planes, int* list_count, uint2* list,
                               int cap, unsigned long long* norm, unsigned* keymax,
                               unsigned long long* norm_max, unsigned* dmax, int64_t group_rows,
                               int64_t group_stride) {
  ResidueOperand o{};
  o.X = X;
  o.ld = ld;
  o.op = op;
  o.rows = rows;
  o.K = K;
  o.Kp = Kp;
  o.emax = emax;
  o.planes = planes;
  o.list_count = list_count;
  o.list = list;
  o.cap = cap;
  o.norm = norm;
  o.keymax = keymax;
  o.norm_max = norm_max;
  o.dmax = dmax;
  o.group_rows = static_cast<int32_t>(group_rows);      // (below 2^30 where grouped)
  o.group_stride = static_cast<int32_t>(group_stride);  // (below 2^31 where grouped)
  return o;
}
// 64-row blocks of A plus 64-row blocks of B's per-row arrays (a strided
// batch's entries have N a multiple of 64, so no block spans two entries)
int64_t tiles_mn(const GemmArgs& g) {
  return (g.M + kTile - 1) / kTile + (rows_of_b(g) + kTile - 1) / kTile;
}

}  // namespace

size_t scratch_bytes(const GemmArgs& g, int64_t slots) {
  const int64_t tiles = ((g.M + kTile - 1) / kTile) * ((g.N + kTile - 1) / kTile);
  const int64_t nb = rows_of_b(g);
  size_t b = align_up(sizeof(int) * size_t(g.M + nb), 256);         // emax
  b += align_up(sizeof(int) * size_t(g.M + nb), 256);               // deep
  b += align_up(size_t(tiles), 256);                                 // route
  b += align_up(sizeof(int) * size_t(tiles + 1), 256);              // general-tile list
  b += align_up(sizeof(int) * size_t(tiles_mn(g)), 256);            // block maxima
  if (g.P == nullptr) b += sizeof(int64_t) * size_t(slots) * kPlanes * kTile * kTile;
  return b;
}

Scratch carve_scratch(void* base, const GemmArgs& g, int64_t slots) {
  const int64_t tiles = ((g.M + kTile - 1) / kTile) * ((g.N + kTile - 1) / kTile);
  char* p = static_cast<char*>(base);
  Scratch s{};
  const int64_t nb = rows_of_b(g);
  s.emaxA = reinterpret_cast<int*>(p);
  s.emaxB = s.emaxA + g.M;
  p += align_up(sizeof(int) * size_t(g.M + nb), 256);
  s.deepA = reinterpret_cast<int*>(p);
  s.deepB = s.deepA + g.M;
  p += align_up(sizeof(int) * size_t(g.M + nb), 256);
  s.route = reinterpret_cast<uint8_t*>(p);
  p += align_up(size_t(tiles), 256);
  s.general = reinterpret_cast<int*>(p);
  p += align_up(sizeof(int) * size_t(tiles + 1), 256);
  s.bmax = reinterpret_cast<int*>(p);
  p += align_up(sizeof(int) * size_t(tiles_mn(g)), 256);
  s.fallback = g.P == nullptr ? reinterpret_cast<int64_t*>(p) : nullptr;
  s.slots = slots;
  return s;
}

cudaError_t run_gemm_with_scratch(const GemmArgs& g, void* scratch, int64_t slots,
                                  bool allow_alloc, cudaStream_t stream) {
  const Scratch s = carve_scratch(scratch, g, slots);
  cudaError_t e;
  {
    StageScope t(kStagePrepass, stream);
    e = launch_prepass(g, s, stream);
  }
  if (e != cudaSuccess) return e;
  {
    StageScope t(kStageBand, stream);
    e = launch_band(g, s, stream);
  }
  if (e != cudaSuccess) return e;
  StageScope t(kStageGeneral, stream);
  return launch_kulisch(g, s.general, allow_alloc, stream);
}

cudaError_t pool_alloc(void** p, size_t bytes, cudaStream_t stream) {
  cudaMemPool_t pool;
  cudaError_t e = device_pool(&pool);
  if (e != cudaSuccess) return e;
  g_pool_allocs.fetch_add(1, std::memory_order_relaxed);
  return cudaMallocFromPoolAsync(p, bytes, pool, stream);
}

cudaError_t pool_stats(uint64_t* allocations, uint64_t* reserved, uint64_t* used) {
  if (allocations != nullptr) *allocations = g_pool_allocs.load(std::memory_order_relaxed);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lock(g_pool_mu);
    pool = g_pool[dev];
  }
  uint64_t r = 0, u = 0;
  if (pool != nullptr) {
    e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &r);
    if (e == cudaSuccess) e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemCurrent, &u);
    if (e != cudaSuccess) return e;
  }
  if (reserved != nullptr) *reserved = r;
  if (used != nullptr) *used = u;
  return cudaSuccess;
}

cudaError_t pool_release() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  // every stream-ordered free must have run before its memory can go back
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  return g_pool[dev] != nullptr ? cudaMemPoolTrimTo(g_pool[dev], 0) : cudaSuccess;
}

cudaError_t pool_set_retention(uint64_t bytes) {
  std::lock_guard<std::mutex> lock(g_pool_mu);
  g_retention = bytes;
  for (int d = 0; d < kMaxDevices; ++d) {
    if (g_pool[d] == nullptr) continue;
    uint64_t keep = bytes;
    const cudaError_t e = cudaMemPoolSetAttribute(g_pool[d], cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace {

cudaError_t launch_band_path(const GemmArgs& g, cudaStream_t stream) {
  const int64_t slots = band_slots(g);
  void* scratch = nullptr;
  cudaError_t e = pool_alloc(&scratch, scratch_bytes(g, slots), stream);
  if (e != cudaSuccess) return e;
  e = run_gemm_with_scratch(g, scratch, slots, true, stream);
  cudaError_t f = cudaFreeAsync(scratch, stream);
  return e != cudaSuccess ? e : f;
}

constexpr int kMaxBands = 4;
std::atomic<int> g_wide_path{1};                   // det_set_wide_path

struct ResidueScratch {
  size_t bytes;
  size_t off_counts, off_norms, zero_bytes, off_deep_idx, off_listA, off_listB, off_planesA,
      off_planesB, off_res;
};

ResidueScratch residue_layout(const GemmArgs& g, int nplanes, int64_t Kp, int cap) {
  ResidueScratch r{};
  size_t b = align_up(scratch_bytes(g, 0), 1024);
  // zeroed together: countA [M], countB [N], error, deep-row/col counters [2],
  // moduli per band [kMaxBands], fused-launch block counters [kMaxBands],
  // exponent-key maxima keymaxA [M], keymaxB [N], the largest deep count of
  // every 64-row block of A and of B [tiles_m + tiles_n]; then the row-norm
  // bounds normA [M], normB [N] and four slots per band [4 kMaxBands] (norm
  // maxima of A and B, and the moduli kernel's two block minima)
  // (B's per-row arrays have rows_of_b rows: every entry's of a strided batch)
  const int64_t nb = rows_of_b(g);
  r.off_counts = b;
  r.off_norms = align_up(b + sizeof(int) * size_t(2 * (g.M + nb) + 3 + 2 * kMaxBands +
                                                  tiles_mn(g)), 8);
  b = r.off_norms + sizeof(unsigned long long) * size_t(g.M + nb + 4 * kMaxBands);
  r.zero_bytes = b - r.off_counts;
  b = align_up(b, 1024);
  r.off_deep_idx = b;                    // deep rows [M], deep columns [N]
  b = align_up(b + sizeof(int) * size_t(g.M + nb), 1024);
  r.off_listA = b;
  b = align_up(b + sizeof(uint2) * size_t(g.M) * cap, 1024);
  r.off_listB = b;
  b = align_up(b + sizeof(uint2) * size_t(nb) * cap, 1024);
  r.off_planesA = b;
  b = align_up(b + size_t(2) * nplanes * size_t(plane_rows(g.M)) * size_t(Kp), 1024);
  r.off_planesB = b;
  b = align_up(b + size_t(2) * nplanes * size_t(plane_rows(nb)) * size_t(Kp), 1024);
  r.off_res = b;
  b = align_up(b + size_t(nplanes) * size_t(g.M) * size_t(g.N), 1024);
  r.bytes = b;
  return r;
}

// Banded schedule.  C is cut into row bands; band b's tensor-core GEMM runs on
// a high-priority library stream while the caller's stream computes the next
// band's A residue planes and the previous band's reconstruction, so the
// CUDA-core stages overlap the tensor-core kernel.  A band's outputs with
// deep elements are reconstructed on a second library stream beside its
// other outputs (that kernel mostly waits on memory).  Only stream order and
// events connect the streams (no kernel waits on another).
struct BandSync {
  cudaStream_t hi = nullptr;                       // tensor-core launches of even bands
  cudaStream_t hi2 = nullptr;                      // ... and of odd bands
  cudaStream_t side = nullptr;                     // deep-output reconstruction
  cudaStream_t gen = nullptr;                      // general-tile kernel
  cudaStream_t fast2 = nullptr;                    // fast reconstruction of bands >= 1
  cudaStream_t wide = nullptr;                     // general tiles: statistics and planes
  cudaEvent_t gen_fork = nullptr, gen_done = nullptr;   // after the routing; general kernel done
  cudaEvent_t wide_planes = nullptr, wide_gemm = nullptr;  // gen -> tensor-core stream -> gen
  cudaEvent_t planes_done[kMaxBands] = {};         // caller's stream -> hi
  cudaEvent_t gemm_done[kMaxBands] = {};           // hi -> caller's stream
  cudaEvent_t deep_done[kMaxBands] = {};           // side -> caller's stream
  cudaEvent_t fast_done[kMaxBands] = {};           // fast2 -> caller's stream
};
std::mutex g_band_mu[kMaxDevices];
BandSync g_band[kMaxDevices];

cudaError_t band_sync(int dev, BandSync** out) {
  BandSync& b = g_band[dev];
  if (b.hi == nullptr) {
    int least = 0, greatest = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    cudaStream_t hi = nullptr;
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&hi, cudaStreamNonBlocking, greatest);
    if (e == cudaSuccess && b.hi2 == nullptr)
      e = cudaStreamCreateWithPriority(&b.hi2, cudaStreamNonBlocking, greatest);
    // the deep kernel's few blocks go ahead of the caller's kernels, behind
    // the tensor-core launches
    const int side_prio = greatest < least ? greatest + 1 : greatest;
    if (e == cudaSuccess && b.side == nullptr)
      e = cudaStreamCreateWithPriority(&b.side, cudaStreamNonBlocking, side_prio);
    if (e == cudaSuccess && b.gen == nullptr)
      e = cudaStreamCreateWithPriority(&b.gen, cudaStreamNonBlocking, least);
    // (a priority above the caller's let the last band's reconstruction
    // crowd band 0's: measured slower)
    if (e == cudaSuccess && b.fast2 == nullptr)
      e = cudaStreamCreateWithPriority(&b.fast2, cudaStreamNonBlocking, least);
    // small kernels that fit beside a tensor-core CTA (no shared memory but
    // the planes kernel's, which prefers the largest carveout): dispatched
    // ahead of the reconstruction's many blocks
    if (e == cudaSuccess && b.wide == nullptr)
      e = cudaStreamCreateWithPriority(&b.wide, cudaStreamNonBlocking, greatest);
    if (e == cudaSuccess && b.gen_fork == nullptr)
      e = cudaEventCreateWithFlags(&b.gen_fork, cudaEventDisableTiming);
    if (e == cudaSuccess && b.gen_done == nullptr)
      e = cudaEventCreateWithFlags(&b.gen_done, cudaEventDisableTiming);
    if (e == cudaSuccess && b.wide_planes == nullptr)
      e = cudaEventCreateWithFlags(&b.wide_planes, cudaEventDisableTiming);
    if (e == cudaSuccess && b.wide_gemm == nullptr)
      e = cudaEventCreateWithFlags(&b.wide_gemm, cudaEventDisableTiming);
    for (int i = 0; i < kMaxBands && e == cudaSuccess; ++i) {
      cudaEvent_t* ev[4] = {&b.planes_done[i], &b.gemm_done[i], &b.deep_done[i], &b.fast_done[i]};
      for (int k = 0; k < 4 && e == cudaSuccess; ++k)
        if (*ev[k] == nullptr) e = cudaEventCreateWithFlags(ev[k], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
      if (hi != nullptr) cudaStreamDestroy(hi);
      return e;
    }
    b.hi = hi;
  }
  *out = &b;
  return cudaSuccess;
}

// Row bands: two bands of whole 256-row tiles once each still fills the GPU
// with tensor-core work.  Band 0's reconstruction runs beside band 1's GEMM,
// band 1's after the last GEMM; a GEMM's time grows with K and a
// reconstruction's does not, so the longer K, the larger band 0.  Measured
// with the two GEMMs on two streams: at 4096 x 4096, 8 + 8 tiles were best
// for K = 2048 and 11 + 5 for K = 4096 (8 + 8: 1.5 % slower; 3 or 4 bands:
// 1.5-6 % slower); at 2048 x 4096 x 4096, 5 + 3.
int band_bounds(const GemmArgs& g, int64_t (&edge)[kMaxBands + 1]) {
  edge[0] = 0;
  if (g.M < 2048) {
    edge[1] = g.M;
    return 1;
  }
  // a strided batch is cut between entries (each band's GEMM takes whole
  // entries); one entry of 2048 rows or more stays one band
  const int64_t unit = g.batch > 1 ? g.Me : 256;
  const int64_t tiles = (g.M + unit - 1) / unit;
  if (tiles < 2) {
    edge[1] = g.M;
    return 1;
  }
  double f = 0.5 + 0.19 * log2(static_cast<double>(g.K) / 2048.0);
  f = f < 0.5 ? 0.5 : (f > 0.69 ? 0.69 : f);
  int64_t t0 = static_cast<int64_t>(static_cast<double>(tiles) * f);
  t0 = t0 < 1 ? 1 : (t0 > tiles - 1 ? tiles - 1 : t0);
  edge[1] = t0 * unit;
  edge[2] = g.M;
  return 2;
}

cudaError_t run_residue_path(const GemmArgs& g, char* base, const ResidueScratch& L, int nplanes,
                             int64_t Kp, int cap, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_band_mu[dev]);     // the streams and events are shared
  BandSync* bs = nullptr;
  e = band_sync(dev, &bs);
  if (e != cudaSuccess) return e;
  const cudaStream_t hi = bs->hi;
  // band b's GEMM on hi (even b) or hi2 (odd b): the next band's CTA pairs
  // take the SMs that the previous band's pairs leave as they finish, instead
  // of waiting for its last pair (a band's work rarely divides evenly among
  // the pairs)
  auto hi_of = [&](int b) { return (b & 1) ? bs->hi2 : hi; };

  unsigned* status = nullptr;                     // sticky expiry record of the TC kernels
  e = device_status_word(&status);
  if (e != cudaSuccess) return e;
  const Scratch s = carve_scratch(base, g, 0);
  int* counts = reinterpret_cast<int*>(base + L.off_counts);
  const int64_t nbr = rows_of_b(g);                                  // B's per-row arrays
  int* error = counts + g.M + nbr;
  int* used = error + 3;                                             // moduli per band
  unsigned* done = reinterpret_cast<unsigned*>(used + kMaxBands);    // fused-launch counters
  unsigned* keymax = done + kMaxBands;                               // [M] then [N]
  unsigned* dmax = keymax + g.M + nbr;                               // [tiles_m] then B's blocks
  const int64_t tiles_m = (g.M + kTile - 1) / kTile, blocks_b = (nbr + kTile - 1) / kTile;
  unsigned long long* norms = reinterpret_cast<unsigned long long*>(base + L.off_norms);
  unsigned long long* maxima = norms + g.M + nbr;                    // [4 b]: band b's A, [1]: B
  const int least = residue_planes_least(g.bf16);
  uint2* listA = reinterpret_cast<uint2*>(base + L.off_listA);
  uint2* listB = reinterpret_cast<uint2*>(base + L.off_listB);
  __nv_bfloat16* planesA = reinterpret_cast<__nv_bfloat16*>(base + L.off_planesA);
  __nv_bfloat16* planesB = reinterpret_cast<__nv_bfloat16*>(base + L.off_planesB);
  int8_t* res = reinterpret_cast<int8_t*>(base + L.off_res);
  int* deep_rows = reinterpret_cast<int*>(base + L.off_deep_idx);   // [M] rows, then [N] columns
  int64_t edge[kMaxBands + 1];
  const int nb = band_bounds(g, edge);
  note_moduli_bands(nb);
  const int64_t nkb = Kp / kStageK;
  const size_t es = g.bf16 ? 2 : 4;

  // K-contiguous, aligned operands with K <= kFusedK take the fused kernel:
  // exponent maxima, planes, norms and the moduli count in one launch per
  // band (no separate pre-pass over A and B)
  // (a strided batch: B's operand is every entry's rows, stacked)
  const bool grouped = g.batch > 1;
  const ResidueOperand rb = residue_operand(g.B, g.ldb, g.opB, nbr, g.K, Kp, s.emaxB, planesB,
                                             counts + g.M, listB, cap, norms + g.M, keymax + g.M,
                                             maxima + 1, dmax + tiles_m, grouped ? g.N : 0,
                                             grouped ? g.strideB : 0);
  const ResidueOperand whole_a = residue_operand(g.A, g.lda, g.opA, g.M, g.K, Kp, nullptr, nullptr,
                                                 nullptr, nullptr, 0, nullptr, nullptr, nullptr,
                                                 nullptr, grouped ? g.Me : 0,
                                                 grouped ? g.strideA : 0);
  const bool fused = fused_residues_ok(rb, g.bf16) && fused_residues_ok(whole_a, g.bf16);
  if (grouped && !fused) return cudaErrorInvalidValue;   // the caller checks batched_residue_ok
  {
    StageScope t(kStagePrepass, stream);
    e = fused ? cudaSuccess : launch_emax(g, s, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(counts, 0, L.zero_bytes, stream);
  }
  if (e != cudaSuccess) return e;
  const ModuliThresholds thr = moduli_thresholds(g.bf16);
  auto fused_band = [&](int b) {
    const int64_t m0 = edge[b], rows = edge[b + 1] - edge[b];
    return FusedBand{maxima + 4 * b, maxima + 1, done + b, used + b, b, least, nplanes, thr,
                     dmax + m0 / kTile, (rows + kTile - 1) / kTile, dmax + tiles_m, blocks_b,
                     deep_list_cap(g.K)};
  };
  // the residue kernels' deep-list counters double as the rows' deep counts,
  // from which the tiles are routed
  auto operand_of_band = [&](int b) {
    const int64_t m0 = edge[b], rows = edge[b + 1] - edge[b];
    // (a strided batch's bands start on an entry: rows m0.. are entry m0 / Me's)
    const void* X = static_cast<const char*>(g.A) +
                    (grouped ? (m0 / g.Me) * g.strideA : (g.opA ? m0 : m0 * g.lda)) * es;
    return residue_operand(X, g.lda, g.opA, rows, g.K, Kp, s.emaxA + m0,
                           planesA + (m0 / kPlaneRows) * nkb * nplanes * kPlaneRows * kStageK,
                           counts + m0, listA + m0 * cap, cap, norms + m0, keymax + m0,
                           maxima + 4 * b, dmax + m0 / kTile, grouped ? g.Me : 0,
                           grouped ? g.strideA : 0);
  };
  // the band's moduli count, once its rows' and B's norm bounds are complete
  auto moduli_of_band = [&](int b) {
    return launch_moduli(norms + edge[b], edge[b + 1] - edge[b], norms + g.M, nbr, g.bf16, least,
                         nplanes, used + b, b, maxima + 4 * b, counts + edge[b], counts + g.M,
                         deep_list_cap(g.K), stream);
  };
  auto planes_of_band = [&](int b) {
    const ResidueOperand oa = operand_of_band(b);
    if (fused) return launch_residues_fused(oa, nullptr, g.bf16, nplanes, fused_band(b), stream);
    cudaError_t ep = launch_residues(oa, g.bf16, nplanes, stream);
    return ep == cudaSuccess ? moduli_of_band(b) : ep;
  };
  auto gemm_of_band = [&](int b) {
    const int64_t m0 = edge[b], rows = edge[b + 1] - edge[b];
    const cudaStream_t hs = hi_of(b);
    StageScope t(kStageResidueGemm, hs);
    ResGemmArgs rg{planesA + (m0 / kPlaneRows) * nkb * nplanes * kPlaneRows * kStageK, planesB,
                   rows, g.N, Kp, nplanes, res + m0 * g.N, g.M * g.N, error, status, used + b, least};
    if (grouped) {                         // the band's entries: only their own tiles
      rg.entry_rows = g.Me;
      rg.entry0 = m0 / g.Me;
    }
    // 256 x 256 tiles on CTA pairs, unless a single 128-row tile covers M or
    // the device cannot run clusters of two
    if (rows > 128) {
      const cudaError_t ep = launch_residue_gemm_pair(rg, hs);
      if (ep != cudaErrorNotSupported) return ep;
    }
    return launch_residue_gemm(rg, hs);
  };
  {
    StageScope t(kStageResiduePlanes, stream);
    // B's planes and band 0's A planes in one launch
    const ResidueOperand oa = operand_of_band(0);
    if (fused) {
      e = launch_residues_fused(rb, &oa, g.bf16, nplanes, fused_band(0), stream);
    } else {
      e = launch_residues2(rb, oa, g.bf16, nplanes, stream);
      if (e == cudaSuccess) e = moduli_of_band(0);
    }
  }
  if (e == cudaSuccess) e = cudaEventRecord(bs->planes_done[0], stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hi_of(0), bs->planes_done[0], 0);
  if (e == cudaSuccess) e = gemm_of_band(0);
  if (e == cudaSuccess) e = cudaEventRecord(bs->gemm_done[0], hi_of(0));
  // the later bands' planes, then the routing and the wide path's first
  // half, and only then the later bands' GEMMs: a GEMM launch that is ready
  // but waits for the SMs of band 0's GEMM would keep the routing and those
  // small kernels from being dispatched until band 0's GEMM ended, and every
  // band after the first starts only then anyway.  (With one band, its GEMM
  // is enqueued at once and the wide path's kernels run beside it.)
  for (int b = 1; b < nb && e == cudaSuccess; ++b) {
    {
      StageScope t(kStageResiduePlanes, stream);
      e = planes_of_band(b);
    }
    if (e == cudaSuccess) e = cudaEventRecord(bs->planes_done[b], stream);
  }
  if (e == cudaSuccess) {
    StageScope t(kStageResiduePlanes, stream);
    e = launch_classify(g, counts, counts + g.M, s, deep_rows, deep_rows + g.M, error + 1, stream);
  }
  bool gen_forked = false;
  WidePlan plan{};
  // (a strided batch's general tiles go to the general kernel)
  const bool wide_on = g_wide_path.load(std::memory_order_relaxed) != 0 && !grouped;
  if (e == cudaSuccess && !wide_on) {
    // the wide path switched off: the general kernel takes every general
    // tile, beside the GEMMs on the lowest-priority stream
    e = cudaEventRecord(bs->gen_fork, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(bs->gen, bs->gen_fork, 0);
    if (e == cudaSuccess) {
      gen_forked = true;
      StageScope t(kStageGeneral, bs->gen);
      e = launch_kulisch(g, s.general, true, bs->gen);
    }
    if (e == cudaSuccess) e = cudaEventRecord(bs->gen_done, bs->gen);
  }
  if (e == cudaSuccess && wide_on) {
    // the general tiles need only the routing: the wide path's statistics,
    // norms and planes run on a greatest-priority stream of their own (small
    // kernels that fit beside a tensor-core CTA); its tensor-core GEMM, its
    // reconstruction and the general kernel follow the last band's GEMM on
    // that GEMM's stream: they need whole SMs, and a launch waiting for them
    // any earlier at that priority would hold up the dispatch of the
    // reconstruction.  With no general tile every one of them returns at once.
    e = cudaEventRecord(bs->gen_fork, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(bs->wide, bs->gen_fork, 0);
    if (e == cudaSuccess) {
      gen_forked = true;
      e = wide_prepare(g, s, bs->wide, bs->wide_planes, &plan);
    }
  }
  for (int b = 1; b < nb && e == cudaSuccess; ++b) {
    e = cudaStreamWaitEvent(hi_of(b), bs->planes_done[b], 0);
    if (e == cudaSuccess && wide_on) e = cudaStreamWaitEvent(hi_of(b), bs->wide_planes, 0);
    if (e == cudaSuccess) e = gemm_of_band(b);
    if (e == cudaSuccess) e = cudaEventRecord(bs->gemm_done[b], hi_of(b));
  }
  if (e == cudaSuccess && gen_forked && wide_on) {
    e = wide_finish(g, plan, hi_of(nb - 1), bs->wide_planes);
    if (e == cudaSuccess) e = cudaEventRecord(bs->gen_done, hi_of(nb - 1));
  }
  // Band b's reconstruction needs the routing (gen_fork, recorded on the
  // caller's stream after it) and band b's GEMM.  Its deep outputs go to the
  // side stream; its other outputs to the caller's stream for band 0 and to
  // fast2 for later bands, so that the last band's starts when its GEMM ends
  // even while band 0's is still running.  For det_gemm_partial the fast
  // kernel writes whole row segments (placeholders in the deep columns), so
  // the deep kernel's deep-column part follows it (its deep-row part, which
  // the fast kernel leaves alone, runs beside it).
  const bool cols_after = g.P != nullptr;
  auto recon_args = [&](int b) {
    return ReconArgs{res, nplanes, s.emaxA, s.emaxB, s.route, counts, listA, counts + g.M, listB,
                     cap, error, edge[b], edge[b + 1], used + b};
  };
  auto deep = [&](int b, int parts, int blocks_per_sm) {
    // deep-row/column lists, and their two counters right after the error flag
    StageScope t(kStageReconstruct, bs->side);
    return launch_reconstruct_deep(g, recon_args(b), deep_rows, error + 1, parts, blocks_per_sm,
                                   bs->side);
  };
  int forked = 0, fast_forked = 0;
  for (int b = 0; b < nb && e == cudaSuccess; ++b) {
    e = cudaStreamWaitEvent(bs->side, bs->gen_fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(bs->side, bs->gemm_done[b], 0);
    const cudaStream_t fs = b == 0 ? stream : bs->fast2;
    if (e == cudaSuccess && b > 0) e = cudaStreamWaitEvent(fs, bs->gen_fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(fs, bs->gemm_done[b], 0);
    if (e != cudaSuccess) break;
    forked = b + 1;
    e = deep(b, cols_after ? kDeepRows : kDeepRows | kDeepCols, 1);
    if (e == cudaSuccess && !cols_after) e = cudaEventRecord(bs->deep_done[b], bs->side);
    if (e == cudaSuccess) {
      StageScope t(kStageReconstruct, fs);
      e = launch_reconstruct_fast(g, recon_args(b), fs);
    }
    if (e == cudaSuccess && (b > 0 || cols_after)) {
      e = cudaEventRecord(bs->fast_done[b], fs);
      if (e == cudaSuccess && b > 0) fast_forked = b + 1;
    }
  }
  // det_gemm_partial: every band's deep-row part is enqueued ahead of the
  // deep-column parts, which wait for their band's fast kernel
  for (int b = 0; cols_after && b < forked && e == cudaSuccess; ++b) {
    e = cudaStreamWaitEvent(bs->side, bs->fast_done[b], 0);
    if (e == cudaSuccess) e = deep(b, kDeepCols, 2);
    if (e == cudaSuccess) e = cudaEventRecord(bs->deep_done[b], bs->side);
  }
  for (int b = 0; b < forked && e == cudaSuccess; ++b) e = cudaStreamWaitEvent(stream, bs->deep_done[b], 0);
  for (int b = 1; b < fast_forked && e == cudaSuccess; ++b)
    e = cudaStreamWaitEvent(stream, bs->fast_done[b], 0);
  if (e == cudaSuccess && gen_forked) e = cudaStreamWaitEvent(stream, bs->gen_done, 0);
  if (e != cudaSuccess) {
    // keep the caller's stream ordered after everything enqueued on hi, hi2, side, fast2 and gen
    cudaEvent_t join = bs->gemm_done[0];
    if (cudaEventRecord(join, hi) == cudaSuccess) cudaStreamWaitEvent(stream, join, 0);
    if (cudaEventRecord(join, bs->hi2) == cudaSuccess) cudaStreamWaitEvent(stream, join, 0);
    join = bs->deep_done[0];
    if (cudaEventRecord(join, bs->side) == cudaSuccess) cudaStreamWaitEvent(stream, join, 0);
    join = bs->fast_done[0];
    if (cudaEventRecord(join, bs->fast2) == cudaSuccess) cudaStreamWaitEvent(stream, join, 0);
    if (cudaEventRecord(bs->gen_done, bs->gen) == cudaSuccess) cudaStreamWaitEvent(stream, bs->gen_done, 0);
    if (cudaEventRecord(bs->gen_done, bs->wide) == cudaSuccess) cudaStreamWaitEvent(stream, bs->gen_done, 0);
  }
  return e;
}

}  // namespace

int set_wide_path(int enable) { return g_wide_path.exchange(enable ? 1 : 0); }

bool batched_residue_ok(const GemmArgs& g) {
  if (g.batch <= 1 || g.Me <= 0 || g.M != int64_t(g.batch) * g.Me || g.P != nullptr || g.C == nullptr)
    return false;
  // whole 64-row blocks per entry (routing, tiles), K-contiguous rows for the
  // fused planes kernel, every stacked row index an int
  if (g.Me % kTile != 0 || g.N % kTile != 0 || g.opA != 0 || g.opB != 0 || g.K <= 0) return false;
  if (g.M > (int64_t(1) << 30) || rows_of_b(g) > (int64_t(1) << 30)) return false;
  if (g.strideA < 0 || g.strideB < 0 || g.strideC < 0) return false;
  if (residue_planes_needed(g) <= 0) return false;
  const ResidueOperand a = residue_operand(g.A, g.lda, g.opA, g.M, g.K, 0, nullptr, nullptr, nullptr,
                                           nullptr, 0, nullptr, nullptr, nullptr, nullptr, g.Me,
                                           g.strideA);
  const ResidueOperand b = residue_operand(g.B, g.ldb, g.opB, rows_of_b(g), g.K, 0, nullptr, nullptr,
                                           nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr,
                                           static_cast<int32_t>(g.N), g.strideB);
  return fused_residues_ok(a, g.bf16) && fused_residues_ok(b, g.bf16);
}

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  // a strided batch as one problem only where every stage handles it
  if (g.batch > 1 && !batched_residue_ok(g)) return cudaErrorInvalidValue;
  const int nplanes = residue_planes_needed(g);
  // grid limits: the residue kernel puts 32-row blocks, the tensor-core
  // kernel 128-row tiles, in gridDim.y (at most 65535)
  const bool residue_ok = g.K > 0 && nplanes > 0 && (g.M + 31) / 32 <= 65535 &&
                          (g.N + 31) / 32 <= 65535;
  if (!residue_ok) return launch_band_path(g, stream);
  const int64_t Kp = (g.K + kStageK - 1) / kStageK * kStageK;
  const int cap = deep_list_cap(g.K);
  const ResidueScratch L = residue_layout(g, nplanes, Kp, cap);
  void* scratch = nullptr;
  cudaError_t e = pool_alloc(&scratch, L.bytes, stream);
  if (e != cudaSuccess) return e;
  e = run_residue_path(g, static_cast<char*>(scratch), L, nplanes, Kp, cap, stream);
  cudaError_t f = cudaFreeAsync(scratch, stream);
  return e != cudaSuccess ? e : f;
}

}  // namespace det
