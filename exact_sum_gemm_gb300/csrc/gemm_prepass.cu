// Exponent pre-pass of the exact GEMM, and per-tile routing.
//
// For every row r of an operand (a row of A, or a row of B = a column of C):
//   emax[r] = the largest exponent e (weight of the last significand bit, see
//             det_arith.cuh) over the row's nonzero finite elements;
//   deep[r] = how many elements are non-finite or lie more than kDeepGap
//             binades below emax[r] ("deep" elements).
// The residue path turns the other ("shallow") elements into integers on a
// common per-row grid and handles deep elements one by one from short
// per-row lists of capacity `cap`; the band kernel anchors each output's
// register window at emax_A + emax_B.  A 64x64 output tile whose worst row
// plus worst column hold more than `cap` deep elements is routed to the
// general kernel instead.  Routing changes speed only: every kernel returns
// the same exact digits.
#include <cuda_runtime.h>
#include <stdint.h>

#include "det_arith.cuh"
#include "det_gemm_internal.cuh"
#include "det_kernels.h"

namespace det {
namespace {

constexpr int kThreads = 256;
constexpr int kRowChunk = kThreads * 16;     // op 0: elements of one row per block
constexpr int kColChunk = 64;                // op 1: k values per block

struct StatOperand {
  const void* X;
  int64_t ld;
  int op;
  int64_t rows;
  int* emax;
  int* deep;
  int64_t blocks;
};

__device__ __forceinline__ int row_emax(const int* emax, int64_t r) {
  const int v = emax[r];
  return v == kEmaxEmpty ? 0 : v;
}

// emax of one full kRowChunk of a K-contiguous row whose chunk start is
// 16-byte aligned: 16-byte loads, exponent keys only.
template <int kBf16>
__device__ void emax_chunk_vec(const StatOperand& o, int64_t r, int64_t k0) {
  constexpr int kPer = kBf16 ? 8 : 4;                     // elements per 16-byte load
  constexpr int kLoads = kRowChunk / kPer / kThreads;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(o.X) +
                                                    (r * o.ld + k0) * (kBf16 ? 2 : 4));
  const int tid = threadIdx.x;
  uint4 v[kLoads];
#pragma unroll
  for (int u = 0; u < kLoads; ++u) v[u] = __ldg(src + u * kThreads + tid);
  int key = 0;
#pragma unroll
  for (int u = 0; u < kLoads; ++u) {
    const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (kBf16) {
        key = max(key, max(exp_key(w[q] << 16), exp_key(w[q] & 0xFFFF0000u)));
      } else {
        key = max(key, exp_key(w[q]));
      }
    }
  }
  __shared__ int red[kThreads / 32];
  key = __reduce_max_sync(0xFFFFFFFFu, key);
  if ((tid & 31) == 0) red[tid >> 5] = key;
  __syncthreads();
  if (tid == 0) {
    int k = red[0];
    for (int w = 1; w < kThreads / 32; ++w) k = max(k, red[w]);
    if (k != 0) atomicMax(o.emax + r, k - 150);
  }
}

// pass 0: emax; pass 1: deep counts (needs emax complete)
template <int kBf16, int kPass>
__device__ void stat_block(const StatOperand& o, int64_t K, int64_t b) {
  const int tid = threadIdx.x;
  if (o.op == 0 && kPass == 0) {
    const int64_t nkc = (K + kRowChunk - 1) / kRowChunk;
    const int64_t r = b / nkc;
    const int64_t k0 = (b - r * nkc) * kRowChunk;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(o.X) + (r * o.ld + k0) * (kBf16 ? 2 : 4);
    if (k0 + kRowChunk <= K && (addr & 15u) == 0) {
      emax_chunk_vec<kBf16>(o, r, k0);
      return;
    }
  }
  if (o.op == 0) {
    const int64_t nkc = (K + kRowChunk - 1) / kRowChunk;
    const int64_t r = b / nkc;
    const int64_t k0 = (b - r * nkc) * kRowChunk;
    const int ref = kPass ? row_emax(o.emax, r) - kDeepGap : 0;
    int acc = kPass ? 0 : kEmaxEmpty;
    uint32_t v[kRowChunk / kThreads];
#pragma unroll
    for (int u = 0; u < kRowChunk / kThreads; ++u) {      // all loads in flight at once
      const int64_t k = k0 + u * kThreads + tid;
      v[u] = k < K ? load_bits<kBf16>(o.X, r * o.ld + k) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kRowChunk / kThreads; ++u) {
      const Decoded d = decode_f32_bits(v[u]);
      const bool live = d.m != 0;
      if (kPass) acc += (d.nonfinite || (live && d.e < ref)) ? 1 : 0;
      else acc = live ? max(acc, d.e) : acc;
    }
    __shared__ int red[kThreads / 32];
    acc = kPass ? __reduce_add_sync(0xFFFFFFFFu, acc) : __reduce_max_sync(0xFFFFFFFFu, acc);
    if ((tid & 31) == 0) red[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
      int v = red[0];
      for (int w = 1; w < kThreads / 32; ++w) v = kPass ? v + red[w] : max(v, red[w]);
      if (kPass) {
        if (v) atomicAdd(o.deep + r, v);
      } else if (v != kEmaxEmpty) {
        atomicMax(o.emax + r, v);
      }
    }
  } else {
    const int64_t nrc = (o.rows + kThreads - 1) / kThreads;
    const int64_t kc = b / nrc;
    const int64_t r = (b - kc * nrc) * kThreads + tid;
    if (r >= o.rows) return;
    const int ref = kPass ? row_emax(o.emax, r) - kDeepGap : 0;
    int acc = kPass ? 0 : kEmaxEmpty;
    const int64_t k0 = kc * kColChunk;
#pragma unroll 16
    for (int u = 0; u < kColChunk; ++u) {
      const int64_t k = k0 + u;
      const uint32_t bits = k < K ? load_bits<kBf16>(o.X, k * o.ld + r) : 0u;
      const Decoded d = decode_f32_bits(bits);
      const bool live = d.m != 0;
      if (kPass) acc += (d.nonfinite || (live && d.e < ref)) ? 1 : 0;
      else acc = live ? max(acc, d.e) : acc;
    }
    if (kPass) {
      if (acc) atomicAdd(o.deep + r, acc);
    } else if (acc != kEmaxEmpty) {
      atomicMax(o.emax + r, acc);
    }
  }
}

template <int kBf16, int kPass>
__global__ void __launch_bounds__(kThreads) rowstat_kernel(StatOperand a, StatOperand b, int64_t K) {
  const int64_t blk = blockIdx.x;
  if (blk < a.blocks) stat_block<kBf16, kPass>(a, K, blk);
  else stat_block<kBf16, kPass>(b, K, blk - a.blocks);
}

// Routing, step 1: the largest deep count of every 64-row block of A and of
// every 64-column block of C (one warp each), into bmax[tiles_m + tiles_n].
// With lists (residue path) it also lists the rows of A and columns of C that
// hold deep elements (in any order: every output is computed on its own).
// It resets the general-tile count read by step 2.
__global__ void __launch_bounds__(kThreads) block_max_kernel(const int* deepA, int64_t M,
                                                              const int* deepB, int64_t N, int* bmax,
                                                              int* rows, int* cols, int* nrc,
                                                              int* general) {
  if (blockIdx.x == 0 && threadIdx.x == 0) general[0] = 0;
  const int64_t tiles_m = (M + kTile - 1) / kTile, tiles_n = (N + kTile - 1) / kTile;
  const int64_t w = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= tiles_m + tiles_n) return;                       // whole warps
  const bool is_a = w < tiles_m;
  const int* cnt = is_a ? deepA : deepB;
  const int64_t len = is_a ? M : N;
  const int64_t base = (is_a ? w : w - tiles_m) * kTile;
  int mx = 0;
#pragma unroll
  for (int h = 0; h < kTile / 32; ++h) {
    const int64_t i = base + lane + 32 * h;
    if (i < len) {
      const int c = cnt[i];
      mx = max(mx, c);
      if (rows != nullptr) {
        if (c != 0) {
          if (is_a) rows[atomicAdd(nrc, 1)] = static_cast<int>(i);
          else cols[atomicAdd(nrc + 1, 1)] = static_cast<int>(i);
        }
      }
    }
  }
  mx = __reduce_max_sync(0xFFFFFFFFu, mx);
  if (lane == 0) bmax[w] = mx;
}

// Routing, step 2, one thread per 64x64 tile: 1 = general kernel, 0 = residue
// path / band kernel.  The general kernel's tiles are also listed after a
// count, general[0].  A strided batch (tm_entry > 0 row blocks per entry):
// tile row tm belongs to entry tm / tm_entry, whose column blocks are B's
// blocks from entry * tiles_n on.
__global__ void __launch_bounds__(kThreads) route_kernel(const int* bmax, int64_t tiles_m,
                                                          int64_t tiles_n, int64_t tm_entry, int cap,
                                                          uint8_t* route, int* general) {
  const int64_t tiles = tiles_m * tiles_n;
  for (int64_t t = int64_t(blockIdx.x) * kThreads + threadIdx.x; t < tiles;
       t += int64_t(gridDim.x) * kThreads) {
    const int64_t tm = t / tiles_n, tn = t - (t / tiles_n) * tiles_n;
    const int64_t bn = tm_entry > 0 ? (tm / tm_entry) * tiles_n + tn : tn;
    const bool gen = static_cast<int64_t>(bmax[tm]) + bmax[tiles_m + bn] > cap;
    route[t] = gen ? 1 : 0;
    if (gen) general[1 + atomicAdd(general, 1)] = static_cast<int>(t);
  }
}

StatOperand make_op(const void* X, int64_t ld, int op, int64_t rows, int64_t K, int* emax,
                    int* deep) {
  StatOperand o{X, ld, op, rows, emax, deep, 0};
  if (K == 0 || rows == 0) return o;
  if (op == 0) o.blocks = rows * ((K + kRowChunk - 1) / kRowChunk);
  else o.blocks = ((rows + kThreads - 1) / kThreads) * ((K + kColChunk - 1) / kColChunk);
  return o;
}

template <int kBf16>
cudaError_t rowstat_t(const GemmArgs& g, const Scratch& s, bool deep_pass, cudaStream_t stream) {
  StatOperand a = make_op(g.A, g.lda, g.opA, g.M, g.K, s.emaxA, s.deepA);
  StatOperand b = make_op(g.B, g.ldb, g.opB, g.N, g.K, s.emaxB, s.deepB);
  const int64_t blocks = a.blocks + b.blocks;
  if (blocks > 0) {
    rowstat_kernel<kBf16, 0><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a, b, g.K);
    note_launch();
    if (deep_pass) {
      rowstat_kernel<kBf16, 1><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a, b, g.K);
      note_launch();
    }
  }
  return cudaGetLastError();
}

}  // namespace

int deep_list_cap(int64_t K) {
  const int64_t c = K / 256;
  return static_cast<int>(c > 8 ? c : 8);
}

cudaError_t launch_classify(const GemmArgs& g, const int* deepA, const int* deepB, const Scratch& s,
                            int* deep_rows, int* deep_cols, int* deep_counters,
                            cudaStream_t stream) {
  // (a strided batch: B's blocks are every entry's, N and Me multiples of 64)
  const int64_t nb = rows_of_b(g);
  const int64_t tiles_m = (g.M + kTile - 1) / kTile, tiles_n = (g.N + kTile - 1) / kTile;
  const int64_t warps = tiles_m + (nb + kTile - 1) / kTile;
  const int64_t grid1 = (warps * 32 + kThreads - 1) / kThreads;
  block_max_kernel<<<static_cast<unsigned>(grid1 > 0 ? grid1 : 1), kThreads, 0, stream>>>(
      deepA, g.M, deepB, nb, s.bmax, deep_rows, deep_cols, deep_counters, s.general);
  const int64_t tiles = tiles_m * tiles_n;
  const int64_t grid2 = (tiles + kThreads - 1) / kThreads;
  route_kernel<<<static_cast<unsigned>(grid2 < 1024 ? (grid2 > 0 ? grid2 : 1) : 1024), kThreads, 0,
                 stream>>>(s.bmax, tiles_m, tiles_n, g.batch > 1 ? g.Me / kTile : 0,
                           deep_list_cap(g.K), s.route, s.general);
  note_launch(2);
  return cudaGetLastError();
}

cudaError_t launch_emax(const GemmArgs& g, const Scratch& s, cudaStream_t stream) {
  // emax starts at kEmaxEmpty (every byte 0x80)
  cudaError_t e = cudaMemsetAsync(s.emaxA, 0x80, sizeof(int) * (g.M + g.N), stream);
  if (e != cudaSuccess) return e;
  return g.bf16 ? rowstat_t<1>(g, s, false, stream) : rowstat_t<0>(g, s, false, stream);
}

cudaError_t launch_prepass(const GemmArgs& g, const Scratch& s, cudaStream_t stream) {
  // emax starts at kEmaxEmpty (every byte 0x80), deep counts at 0
  cudaError_t e = cudaMemsetAsync(s.emaxA, 0x80, sizeof(int) * (g.M + g.N), stream);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(s.deepA, 0, sizeof(int) * (g.M + g.N), stream);
  if (e != cudaSuccess) return e;
  e = g.bf16 ? rowstat_t<1>(g, s, true, stream) : rowstat_t<0>(g, s, true, stream);
  if (e != cudaSuccess) return e;
  return launch_classify(g, s.deepA, s.deepB, s, nullptr, nullptr, nullptr, stream);
}

}  // namespace det
