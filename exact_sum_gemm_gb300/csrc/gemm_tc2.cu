// Residue GEMM on CTA pairs: the same exact modular products as
// residue_gemm_kernel (gemm_tc.cu), with 256 x 256 output tiles computed by
// one tcgen05 MMA stream shared by two CTAs on two SMs (cta_group::2).
//
// Why pairs: with one CTA and 128 x 256 tiles, every 64-k stage is written
// into shared memory by TMA and read back by the MMA, 2 x 48 KB per
// 2 x 128 x 256 x 64 flops, which is more shared-memory bandwidth than an SM
// has at the full bf16 rate.  In a pair each CTA stages only its 128 rows of
// A and its half (128 rows) of B, so the same flops move two thirds of the
// bytes through each SM.
//
// Pair layout (cluster of two CTAs, rank 0 = "leader"):
//   * CTA r loads rows m0 + 128r .. of A_u and rows n0 + 128r .. of B_u into
//     its own shared memory; both loads complete on the LEADER's full[s]
//     barrier, whose expected byte count covers both CTAs;
//   * the leader's single MMA thread issues UMMA 256 x 256 x 16 (bf16 ->
//     f32); CTA r's TMEM receives output rows m0 + 128r .. (all 256 columns);
//   * commits are multicast to both CTAs (empty[s], acc_ready[.]); the eight
//     epilogue warps of the pair arrive on the leader's acc_free[.];
//   * each CTA's epilogue reduces its 128 x 256 accumulator modulo p in TMEM
//     every 832 K exactly as the single-CTA kernel does.
// Work: the (modulus, 256 x 256 tile) pairs in modulus-major order, so the
// clusters in flight share few moduli's planes in L2.  Cluster c takes every
// C-th of them from c on (C clusters), two at a time on the two accumulators.
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel records an
// error flag, drains what is in flight and both CTAs meet at a final cluster
// barrier before TMEM is released.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "det_kernels.h"
#include "det_residue.cuh"
#include "tc_ptx.cuh"

namespace det {

bool make_plane_map(CUtensorMap* map, const void* base, int64_t rows, int64_t Kp, int planes,
                    int box_rows);

namespace {

constexpr int kPairM = 256;                                  // output tile rows (both CTAs)
constexpr int kHalfM = 128;                                  // rows per CTA
constexpr int kTileN = 256;
constexpr int kStages = 6;
constexpr int kThreads = 192;
constexpr int kABytes = kHalfM * kStageK * 2;                // 16 KB: this CTA's A rows
constexpr int kBBytes = (kTileN / 2) * kStageK * 2;          // 16 KB: this CTA's half of B
constexpr int kStageBytes = kABytes + kBBytes;               // 32 KB
constexpr int kKbPerChunk = kChunkK / kStageK;               // 13
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kPairM, kTileN);
constexpr int kTmemCols = 512;                               // two 256-column accumulators
constexpr size_t kSmemBytes = size_t(kStages) * kStageBytes + 1024 + 1024;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
static_assert(kHalfM % kPlaneRows == 0 && (kTileN / 2) % kPlaneRows == 0, "whole row groups");

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity) {
  return ptx::mbar_wait_ns(bar, parity, kWaitLimitNs);
}

// A bounded wait ran out: the call's outputs become NaN (per-call flag) and
// the library's device status records the expiry (det_device_status).
__device__ __forceinline__ void report_timeout(const ResGemmArgs& a) {
  atomicExch(a.error, 1);
  if (a.status != nullptr) atomicOr(a.status, kStatusTimeout);
}

__device__ __forceinline__ void job_at(int J, int T, int& tt, int& c) {
  c = J / T;
  tt = J - c * T;
}

template <int kTiling>
__global__ void __launch_bounds__(kThreads, 1)
    residue_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB, ResGemmArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);   // leader's used
  uint64_t* empty = full + kStages;
  uint64_t* acc_ready = empty + kStages;
  uint64_t* acc_free = acc_ready + 2;                                            // leader's used
  uint64_t* fin = acc_free + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fin + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int64_t cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
  const int nkb = static_cast<int>(a.Kp / kStageK);
  const int nch = (nkb + kKbPerChunk - 1) / kKbPerChunk;
  // (a strided batch: each entry's own tiles, or several entries per tile)
  const int64_t pack = gemm_pack<kPairM, kTileN, kTiling>(a);
  const int64_t tiles = kTiling == kTilingListed ? int64_t(a.tile_list[0])    // (the count first)
                                                 : gemm_tiles<kPairM, kTileN, kTiling>(a, pack);
  const int64_t singles = tiles * planes_used(a);  // (modulus, tile), modulus-major
  // a cluster with no item (a launch sized for more moduli than it computes)
  // issues no MMA, so it neither commits nor waits for the final commit
  const bool has_work = cluster < singles;
  if (singles == 0) return;                // nothing for any cluster: leave before any set-up

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&acc_ready[i], 1);
      ptx::mbar_init(&acc_free[i], 8);      // four epilogue warps in each CTA of the pair
    }
    ptx::mbar_init(fin, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_holder, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();                     // both CTAs' barriers initialised
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // The cluster takes singles cluster, cluster + C, cluster + 2C, ... (C
  // clusters), two at a time: unit j interleaves singles cluster + 2jC and
  // cluster + (2j + 1)C on the two accumulators (T = 1 if the second is
  // past the end).  A launch then ends within half a unit of its ideal
  // length, whatever its tile count.
  auto unit_at = [&](int64_t j, int64_t (&sg)[2], int& T) {
    sg[0] = cluster + 2 * j * clusters;
    sg[1] = sg[0] + clusters;
    T = sg[1] < singles ? 2 : 1;
    return sg[0] < singles;
  };
  auto single_at = [&](int64_t sgl, int& u, int64_t& t) {
    u = static_cast<int>(sgl / tiles);
    t = sgl - static_cast<int64_t>(u) * tiles;
  };


  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      uint32_t it = 0;
      const uint32_t full_leader = ptx::map_to_cta(ptx::smem_addr(full), 0);
      for (int64_t j = 0; ok; ++j) {
        int64_t sg[2];
        int T;
        if (!unit_at(j, sg, T)) break;
        for (int J = 0; J < T * nch && ok; ++J) {
          int tt, c, u;
          job_at(J, T, tt, c);
          int64_t t, m0, nb0, n0, m_end;
          single_at(sg[tt], u, t);
          gemm_tile<kPairM, kTileN, kTiling>(a, pack, t, m0, nb0, n0, m_end);
          const int ga = static_cast<int>((m0 + kHalfM * rank) / kPlaneRows);
          const int gb = static_cast<int>((nb0 + (kTileN / 2) * rank) / kPlaneRows);
          const int kb_end = min(nkb, (c + 1) * kKbPerChunk);
          for (int kb = c * kKbPerChunk; kb < kb_end; ++kb) {
            const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
            if (!wait_bounded(&empty[s], ph ^ 1u)) {
              ok = false;
              break;
            }
            if (rank == 0) ptx::mbar_arrive_expect_tx(&full[s], 2 * kStageBytes);
            unsigned char* st = smem + s * kStageBytes;
            const uint32_t bar = full_leader + s * static_cast<uint32_t>(sizeof(uint64_t));
            ptx::tma_load_5d_pair(st, &tmA, bar, 0, 0, u, kb, ga);
            ptx::tma_load_5d_pair(st + kABytes, &tmB, bar, 0, 0, u, kb, gb);
            ++it;
          }
        }
      }
      // drain before the pair may exit.  The leader waits for the last
      // stages' loads of both CTAs (their bytes land on its barriers); each
      // CTA then waits (normal path) for the MMA's release of those stages,
      // whose commits arrive on barriers in its own shared memory.
      const uint32_t first = it > uint32_t(kStages) ? it - kStages : 0u;
      if (rank == 0)
        for (uint32_t j = first; j < it; ++j) wait_bounded(&full[j % kStages], (j / kStages) & 1u);
      if (ok) {
        for (uint32_t j = first; j < it; ++j)
          if (!wait_bounded(&empty[j % kStages], (j / kStages) & 1u)) ok = false;
      }
      if (!ok) report_timeout(a);
    }
  }
  else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      bool ok = true;
      uint32_t it = 0;
      uint32_t uses[2] = {0u, 0u};
      for (int64_t j = 0; ok; ++j) {
        int64_t sg[2];
        int T;
        if (!unit_at(j, sg, T)) break;
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
          const uint32_t tmem_d = tmem_base + static_cast<uint32_t>(acc * kTileN);
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
              ptx::mma_bf16_pair(tmem_d, ad, bd, kIdesc, accumulate);
            }
            ptx::mma_commit_pair(&empty[s]);   // stage s free in both CTAs once these finish
            ++it;
          }
          if (!ok) break;
          ptx::mma_commit_pair(&acc_ready[acc]);   // window c of modulus u in both TMEMs
        }
      }
      if (!ok) report_timeout(a);
      if (has_work) ptx::mma_commit_pair(fin);     // every MMA of this CTA pair has completed
    }
  } else {
    const int g = warp & 3;                // TMEM lanes 32g .. 32g+31 of this CTA
    bool ok = true;
    uint32_t uses[2] = {0u, 0u};
    const uint32_t free_leader = ptx::map_to_cta(ptx::smem_addr(acc_free), 0);
    for (int64_t j = 0; ok; ++j) {
      int64_t sg[2];
      int T;
      if (!unit_at(j, sg, T)) break;
      for (int J = 0; J < T * nch; ++J) {
        int tt, c, u;
        job_at(J, T, tt, c);
        int64_t t, m0, nb0, n0, m_end;
        single_at(sg[tt], u, t);
        gemm_tile<kPairM, kTileN, kTiling>(a, pack, t, m0, nb0, n0, m_end);
        const int64_t row = m0 + kHalfM * rank + 32 * g + lane;
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
        for (int cb = 0; cb < kTileN / 32; ++cb) {
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * g) << 16) +
                                 static_cast<uint32_t>(acc * kTileN + cb * 32);
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
            // a second reduction makes the residue balanced; its byte is the
            // low byte of the pattern of r + 1.5*2^23
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
              packed[j4] = __byte_perm(__byte_perm(b[0], b[1], 0x0040),
                                       __byte_perm(b[2], b[3], 0x0040), 0x5410);
            }
            const int64_t n_left = a.N - col;
            if (n_left >= 32 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
              // evict-first: read once, by the reconstruction after the launch
              __stcs(reinterpret_cast<uint4*>(out), make_uint4(packed[0], packed[1], packed[2], packed[3]));
              __stcs(reinterpret_cast<uint4*>(out) + 1, make_uint4(packed[4], packed[5], packed[6], packed[7]));
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
        if (lane == 0)                               // on the leader's barrier
          ptx::mbar_arrive_cluster(free_leader + static_cast<uint32_t>(acc * sizeof(uint64_t)));
      }
    }
    if (!ok && lane == 0) report_timeout(a);
  }

  // this CTA's roles are done; then every MMA of the pair has finished
  // writing both TMEMs (a short bounded wait: the leader's last commit), and
  // both CTAs meet before the columns are released
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1 && has_work) {
    if (!wait_bounded(fin, 0) && lane == 0) report_timeout(a);
  }
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
}

}  // namespace

cudaError_t launch_residue_gemm_pair(const ResGemmArgs& a, cudaStream_t stream) {
  if (a.M == 0 || a.N == 0 || a.Kp == 0 || a.nplanes <= 0) return cudaSuccess;
  static PerDeviceOnce queried;
  static int max_clusters[kMaxDevices] = {};            // -1: clusters of two unusable
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = queried.run([&](int d) {
    int n = 0, sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
    cudaError_t r = cudaSuccess;
    for (auto kern : {residue_gemm_pair_kernel<kTilingPlain>, residue_gemm_pair_kernel<kTilingEntries>,
                      residue_gemm_pair_kernel<kTilingListed>})
      if (r == cudaSuccess)
        r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3(static_cast<unsigned>(sms > 1 ? sms / 2 * 2 : 2), 1, 1);
    if (r == cudaSuccess)
      r = cudaOccupancyMaxActiveClusters(&n, residue_gemm_pair_kernel<kTilingPlain>, &q);
    max_clusters[d] = (r == cudaSuccess && n > 0) ? n : -1;
    cudaGetLastError();                                 // a failed query is not the caller's error
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e == cudaErrorInvalidDevice ? cudaErrorNotSupported : e;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (max_clusters[dev] < 0) return cudaErrorNotSupported;
  CUtensorMap tmA, tmB;
  if (!make_plane_map(&tmA, a.A, a.M, a.Kp, a.nplanes, kHalfM) ||
      !make_plane_map(&tmB, a.B, gemm_b_rows(a), a.Kp, a.nplanes, kTileN / 2))
    return cudaErrorInvalidValue;
  // (a listed launch: every tile as the bound; its CTAs past the list's work return)
  const int64_t tiles = a.entry_rows > 0
                            ? gemm_tiles<kPairM, kTileN, kTilingEntries>(a, gemm_pack<kPairM, kTileN, kTilingEntries>(a))
                            : gemm_tiles<kPairM, kTileN, kTilingPlain>(a, 1);
  // sized for the fewest moduli the launch may compute, so every cluster
  // has at least one item whatever count the device chooses
  const int64_t singles =
      tiles * (a.grid_moduli > 0 ? a.grid_moduli : (a.used != nullptr ? a.used_min : a.nplanes));
  const int64_t clusters = singles < max_clusters[dev] ? singles : max_clusters[dev];
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  // (a strided batch's band, or a listed launch: their tilings compiled
  // apart, so that plain launches keep their own register allocation)
  switch (tiling_of(a)) {
    case kTilingEntries: e = cudaLaunchKernelEx(&cfg, residue_gemm_pair_kernel<kTilingEntries>, tmA, tmB, a); break;
    case kTilingListed: e = cudaLaunchKernelEx(&cfg, residue_gemm_pair_kernel<kTilingListed>, tmA, tmB, a); break;
    default: e = cudaLaunchKernelEx(&cfg, residue_gemm_pair_kernel<kTilingPlain>, tmA, tmB, a); break;
  }
  note_launch();
  return e;
}

}  // namespace det
