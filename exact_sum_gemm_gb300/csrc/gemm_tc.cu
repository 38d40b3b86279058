// Residue GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// For every modulus p_u (u < nplanes) it computes, exactly,
//     res[u][m][n] = (sum_k A_u[m,k] * B_u[n,k]) mod p_u,
// where A_u, B_u are bf16 planes of residues with |r| <= 138 (see
// residue.cu).  Each product is an integer of magnitude <= 19044, exact in the
// MMA; fp32 accumulation of integers is exact while the running sum stays
// below 2^24, so the accumulator is reduced modulo p_u in TMEM after every
// 832 values of K (832 * 19044 + a reduced carry < 2^24), and the MMA keeps
// accumulating on top of the reduced value.  The result is the exact integer
// dot product modulo p_u; the CRT in residue.cu rebuilds the exact sum.
//
// Structure (persistent, one CTA per SM, looping over units = (modulus, pair
// of neighbouring 128x256 output tiles), modulus-major):
//   warp 0      TMA producer: 64-wide K stages of A_u (128 rows) and B_u (256
//               rows), 128-byte swizzled, 4-stage mbarrier ring (plane
//               layout: det_residue.cuh)
//   warp 1      TMEM allocation (512 columns = two 128x256 f32 accumulators)
//               and the single MMA-issuing thread (UMMA 128x256x16, bf16)
//   warps 2-5   epilogue: tcgen05.ld the accumulator (each warp owns 32 TMEM
//               lanes = 32 rows), reduce modulo p_u with exact fp32
//               arithmetic, tcgen05.st it back (or, after the last chunk,
//               store the residues to global memory)
// A unit's two tiles are interleaved chunk by chunk on the two accumulators,
// so the MMA of one tile overlaps the in-TMEM reduction of the other.
// Every mbarrier wait is bounded (about 2 s): on expiry the kernel records an
// error flag (the reconstruction then emits NaN), drains its copies in flight,
// frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "det_kernels.h"
#include "det_residue.cuh"
#include "tc_ptx.cuh"

namespace det {
namespace {

constexpr int kBlockM = 128;
constexpr int kBlockN = 256;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kABytes = kBlockM * kStageK * 2;               // 16 KB
constexpr int kBBytes = kBlockN * kStageK * 2;               // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;               // 48 KB
constexpr int kKbPerChunk = kChunkK / kStageK;               // 13
static_assert(kBlockM % kPlaneRows == 0 && kBlockN % kPlaneRows == 0, "tiles cover whole row groups");
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBlockM, kBlockN);
constexpr uint32_t kTmemCols = 512;
constexpr size_t kSmemBytes = size_t(kStages) * kStageBytes + 1024 + 1024;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity) {
  return ptx::mbar_wait_ns(bar, parity, kWaitLimitNs);
}

// A bounded wait ran out: the call's outputs become NaN (per-call flag) and
// the library's device status records the expiry (det_device_status).
__device__ __forceinline__ void report_timeout(const ResGemmArgs& a) {
  atomicExch(a.error, 1);
  if (a.status != nullptr) atomicOr(a.status, kStatusTimeout);
}

// Job J of a unit holding T (1 or 2) tiles -> (tile index tt < T, K chunk c):
// the chunks alternate between the unit's tiles (and their accumulators).
__device__ __forceinline__ void job_at(int J, int T, int& tt, int& c) {
  c = J / T;
  tt = J - c * T;
}

template <int kTiling>
__global__ void __launch_bounds__(kThreads, 1)
    residue_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, ResGemmArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_ready = empty + kStages;
  uint64_t* acc_free = acc_ready + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_free + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = static_cast<int>(a.Kp / kStageK);
  const int nch = (nkb + kKbPerChunk - 1) / kKbPerChunk;
  // work units: (modulus, pair of neighbouring output tiles), modulus-major so
  // that the CTAs in flight share one plane of A and one of B in L2
  // (a strided batch: each entry's own tiles, or several entries per tile)
  const int64_t pack = gemm_pack<kBlockM, kBlockN, kTiling>(a);
  const int64_t tiles = kTiling == kTilingListed ? int64_t(a.tile_list[0])    // (the count first)
                                                 : gemm_tiles<kBlockM, kBlockN, kTiling>(a, pack);
  const int64_t tile_pairs = (tiles + 1) / 2;
  const int64_t units = tile_pairs * planes_used(a);
  if (units == 0) return;                  // nothing to compute: leave before any set-up

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&acc_ready[i], 1);
      ptx::mbar_init(&acc_free[i], 4);      // one arrival per epilogue warp
    }
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // unit -> its modulus, first tile and tile count (2, or 1 for an odd last tile)
  auto unit_at = [&](int64_t unit, int& u, int64_t& t0, int& T) {
    u = static_cast<int>(unit / tile_pairs);
    t0 = 2 * (unit - static_cast<int64_t>(u) * tile_pairs);
    T = t0 + 1 < tiles ? 2 : 1;
  };


  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      uint32_t it = 0;
      for (int64_t unit = blockIdx.x; unit < units && ok; unit += gridDim.x) {
      int u, T;
      int64_t t0;
      unit_at(unit, u, t0, T);
      for (int J = 0; J < T * nch && ok; ++J) {
        int tt, c;
        job_at(J, T, tt, c);
        int64_t m0, nb0, n0, m_end;
        gemm_tile<kBlockM, kBlockN, kTiling>(a, pack, t0 + tt, m0, nb0, n0, m_end);
        const int kb_end = min(nkb, (c + 1) * kKbPerChunk);
        for (int kb = c * kKbPerChunk; kb < kb_end; ++kb) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!wait_bounded(&empty[s], ph ^ 1u)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[s], kStageBytes);
          unsigned char* st = smem + s * kStageBytes;
          ptx::tma_load_5d(st, &tmA, &full[s], 0, 0, u, kb, static_cast<int>(m0 / kPlaneRows));
          ptx::tma_load_5d(st + kABytes, &tmB, &full[s], 0, 0, u, kb,
                           static_cast<int>(nb0 / kPlaneRows));
          ++it;
        }
      }
      }
      // drain before the CTA may exit: the copies still in flight, then (on the
      // normal path) the MMA's release of the last stages, whose commits
      // arrive on barriers in this CTA's shared memory
      const uint32_t first = it > uint32_t(kStages) ? it - kStages : 0u;
      for (uint32_t j = first; j < it; ++j) wait_bounded(&full[j % kStages], (j / kStages) & 1u);
      if (ok) {
        for (uint32_t j = first; j < it; ++j) {
          if (!wait_bounded(&empty[j % kStages], (j / kStages) & 1u)) ok = false;
        }
      }
      if (!ok) report_timeout(a);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      uint32_t it = 0;
      uint32_t uses[2] = {0u, 0u};
      for (int64_t unit = blockIdx.x; unit < units && ok; unit += gridDim.x) {
      int u, T;
      int64_t t0;
      unit_at(unit, u, t0, T);
      for (int J = 0; J < T * nch && ok; ++J) {
        int tt, c;
        job_at(J, T, tt, c);
        const int acc = tt;
        if (!wait_bounded(&acc_free[acc], (uses[acc] & 1u) ^ 1u)) {
          ok = false;
          break;
        }
        ++uses[acc];
        ptx::tc_fence_after();
        const uint32_t tmem_d = tmem_base + static_cast<uint32_t>(acc * kBlockN);
        const int kb_begin = c * kKbPerChunk;
        const int kb_end = min(nkb, kb_begin + kKbPerChunk);
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!wait_bounded(&full[s], ph)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_addr(smem + s * kStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int kk = 0; kk < kStageK / 16; ++kk) {
            const uint64_t ad = ptx::smem_desc_sw128(a_addr + kk * 32);
            const uint64_t bd = ptx::smem_desc_sw128(b_addr + kk * 32);
            const uint32_t accumulate = (c > 0 || kb > kb_begin || kk > 0) ? 1u : 0u;
            ptx::mma_bf16(tmem_d, ad, bd, kIdesc, accumulate);
          }
          ptx::mma_commit(&empty[s]);      // stage s is free once these MMAs finish
          ++it;
        }
        if (!ok) break;
        ptx::mma_commit(&acc_ready[acc]);  // chunk c of modulus u is in TMEM
      }
      }
      if (!ok) report_timeout(a);
    }
  } else {
    const int g = warp & 3;                // TMEM lanes 32g .. 32g+31
    bool ok = true;
    uint32_t uses[2] = {0u, 0u};
    for (int64_t unit = blockIdx.x; unit < units && ok; unit += gridDim.x) {
    int u, T;
    int64_t t0;
    unit_at(unit, u, t0, T);
    for (int J = 0; J < T * nch; ++J) {
      int tt, c;
      job_at(J, T, tt, c);
      int64_t m0, nb0, n0, m_end;
      gemm_tile<kBlockM, kBlockN, kTiling>(a, pack, t0 + tt, m0, nb0, n0, m_end);
      const int64_t row = m0 + 32 * g + lane;
      // a packed tile: this row's entry within the tile (only its own columns)
      const int64_t row_entry = pack > 1 ? entry_div(row - m0, a.entry_rows) : 0;
      const int acc = tt;
      if (!wait_bounded(&acc_ready[acc], uses[acc] & 1u)) {
        ok = false;
        break;
      }
      ++uses[acc];
      ptx::tc_fence_after();
      const bool last = c == nch - 1;
      const float p = static_cast<float>(modulus(u));
      const float inv_p = 1.0f / p;
#pragma unroll 1
      for (int cb = 0; cb < kBlockN / 32; ++cb) {
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * g) << 16) +
                               static_cast<uint32_t>(acc * kBlockN + cb * 32);
        uint32_t v[32];
        ptx::tmem_ld32(taddr, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j)      // exact integers below 2^24: |result| < 131
          v[j] = __float_as_uint(near_mod_f32(__uint_as_float(v[j]), p, inv_p));
        if (!last) {
          ptx::tmem_st32(taddr, v);
        } else if (row < m_end &&
                     (pack <= 1 || entry_div(n0 + cb * 32, a.N) == row_entry)) {
          // a second reduction makes the residue balanced (|r| <= 127); its
          // byte is the low byte of the pattern of r + 1.5*2^23
          const int64_t col = n0 + cb * 32 - row_entry * a.N;   // (0 unless packed)
            int8_t* out = a.res + u * a.res_plane + row * a.N + col;
          uint32_t packed[8];
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            uint32_t b[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float r = near_mod_f32(__uint_as_float(v[4 * j4 + h]), p, inv_p);
              b[h] = __float_as_uint(__fadd_rn(r, kRoundMagic));
            }
            packed[j4] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040),
                                     0x5410);
          }
          const int64_t n_left = a.N - col;
          if (n_left >= 32 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
            reinterpret_cast<uint4*>(out)[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            reinterpret_cast<uint4*>(out)[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < n_left) out[j] = static_cast<int8_t>(packed[j / 4] >> (8 * (j % 4)));
          }
        }
      }
      if (!last) ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acc_free[acc]);
    }
    }
    if (!ok && lane == 0) report_timeout(a);
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 5-D map over the planes [rows/32][Kp/64][P][32][64] of bf16 (innermost
// first: 64 k of one stage, row in group, plane, stage, row group).  A box of
// 64 x 32 x 1 x 1 x box_rows/32 is one plane's 64-k stage for box_rows rows:
// box_rows 128-byte rows in shared memory, in row order, 128-byte swizzled,
// as the UMMA descriptors expect.  Row groups past the end read as zero.
bool make_plane_map(CUtensorMap* map, const void* base, int64_t rows, int64_t Kp, int planes,
                    int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t nkb = static_cast<cuuint64_t>(Kp / kStageK);
  const cuuint64_t block = static_cast<cuuint64_t>(kPlaneRows) * kStageK * 2;     // 4 KB
  cuuint64_t dims[5] = {static_cast<cuuint64_t>(kStageK), static_cast<cuuint64_t>(kPlaneRows),
                        static_cast<cuuint64_t>(planes), nkb,
                        static_cast<cuuint64_t>(plane_rows(rows) / kPlaneRows)};
  cuuint64_t strides[4] = {static_cast<cuuint64_t>(kStageK) * 2, block,
                           static_cast<cuuint64_t>(planes) * block,
                           nkb * static_cast<cuuint64_t>(planes) * block};
  cuuint32_t box[5] = {static_cast<cuuint32_t>(kStageK), static_cast<cuuint32_t>(kPlaneRows), 1, 1,
                       static_cast<cuuint32_t>(box_rows / kPlaneRows)};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_residue_gemm(const ResGemmArgs& a, cudaStream_t stream) {
  if (a.M == 0 || a.N == 0 || a.Kp == 0 || a.nplanes <= 0) return cudaSuccess;
  static PerDeviceOnce configured;                 // the attribute is per device
  cudaError_t ce = configured.run([](int) {
    cudaError_t r = cudaSuccess;
    for (auto kern : {residue_gemm_kernel<kTilingPlain>, residue_gemm_kernel<kTilingEntries>,
                      residue_gemm_kernel<kTilingListed>})
      if (r == cudaSuccess)
        r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
    return r;
  });
  if (ce != cudaSuccess) return ce;
  CUtensorMap tmA, tmB;
  if (!make_plane_map(&tmA, a.A, a.M, a.Kp, a.nplanes, kBlockM) ||
      !make_plane_map(&tmB, a.B, gemm_b_rows(a), a.Kp, a.nplanes, kBlockN))
    return cudaErrorInvalidValue;
  // persistent: one CTA per SM (the shared memory and TMEM footprint allow no more)
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  // (a listed launch: every tile as the bound; its CTAs past the list's work return)
  const int64_t tiles = a.entry_rows > 0
                            ? gemm_tiles<kBlockM, kBlockN, kTilingEntries>(a, gemm_pack<kBlockM, kBlockN, kTilingEntries>(a))
                            : gemm_tiles<kBlockM, kBlockN, kTilingPlain>(a, 1);
  // sized for the fewest moduli the launch may compute (every CTA has a unit)
  const int64_t units = (tiles + 1) / 2 *
      (a.grid_moduli > 0 ? a.grid_moduli : (a.used != nullptr ? a.used_min : a.nplanes));
  const unsigned grid = static_cast<unsigned>(units < sms ? units : sms);
  switch (tiling_of(a)) {
    case kTilingEntries: residue_gemm_kernel<kTilingEntries><<<grid, kThreads, kSmemBytes, stream>>>(tmA, tmB, a); break;
    case kTilingListed: residue_gemm_kernel<kTilingListed><<<grid, kThreads, kSmemBytes, stream>>>(tmA, tmB, a); break;
    default: residue_gemm_kernel<kTilingPlain><<<grid, kThreads, kSmemBytes, stream>>>(tmA, tmB, a); break;
  }
  note_launch();
  return cudaGetLastError();
}

}  // namespace det
