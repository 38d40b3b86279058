// Wide residue path: the exact GEMM on tiles whose operands span many binades.
//
// The narrow residue path puts each row of an operand on an integer grid 18
// binades below the row's largest element and lists what lies deeper; a
// 64x64 output tile whose rows hold more deep elements than its lists take
// is routed to the general kernel.  Data with a wide exponent spread (values
// 2^U[-40,40], bf16 with exponents over +-60) sends every tile there.  This
// path takes those tiles back to the tensor cores with a wider grid:
//
//   base[r]  = the smallest last-bit exponent of row r's nonzero elements,
//   X[r,k]   = m * 2^(e - base[r])  (exact integer, |X| < 2^(b + W), with b =
//              24 significand bits for f32, 8 for bf16, W = emax[r] - base[r]),
//   C[m,n]   = RNE_f32( 2^(baseA[m] + baseB[n]) * S ),  S = sum_k XA[m,k] XB[n,k].
//
// A row qualifies when its spread W is at most kWideSpread (f32 88, bf16 124
// binades) and it holds no Inf/NaN; a general tile whose 64 rows of A and 64
// rows of B all qualify is a wide tile, the others stay with the general
// kernel.  S is computed modulo up to 40 pairwise coprime moduli (the narrow
// path's 14, then 2^8 and primes from 193 down to 71): residue planes in
// bf16, the same tcgen05 GEMM as the narrow path, then the CRT sum in up to
// ten 32-bit limbs.  How many moduli: a Cauchy-Schwarz bound, |S| <=
// max ||XA row|| max ||XB row||, from per-row norm bounds summed with upward
// rounding; their product must exceed 2 (1 + 2^-5) times it.  The exact S,
// placed at bit offset baseA + baseB + 298, gives the output's canonical
// digits, rounded once by the same routine as det_finalize (or written out as
// the partial).  Integer addition is exact, so this is the same exact sum as
// every other path of the library (det-train page, "Method").
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <math.h>

#include "det_arith.cuh"
#include "det_gemm_internal.cuh"
#include "det_kernels.h"
#include "det_residue.cuh"

namespace det {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxLimbs = 10;          // 32-bit limbs of S: moduli products below 2^300
constexpr int kWeightBits = 18;        // fixed-point weights of the CRT quotient
constexpr int kNormUnitBits = 40;      // row norms in units of 2^-40

__host__ __device__ constexpr int sig_bits(int bf16) { return bf16 ? 8 : 24; }
__host__ __device__ constexpr int wide_spread(int bf16) { return bf16 ? 124 : 88; }

// Host-side tables of the moduli choice and the limb count of each prefix.
struct WideTables {
  double log2prod[kNumModuliWide + 1];    // log2 of the product of the first P moduli
  int limbs[kNumModuliWide + 1];          // limbs holding S' mod 2^(32 L), |S| < M/2
};

WideTables make_tables() {
  WideTables t{};
  double acc = 0.0;
  t.log2prod[0] = 0.0;
  t.limbs[0] = 1;
  for (int P = 1; P <= kNumModuliWide; ++P) {
    acc += log2(static_cast<double>(modulus(P - 1)));
    t.log2prod[P] = acc;
    int L = 1;
    while (32.0 * L - 1.0 < acc + 1.0) ++L;      // 2^(32L - 1) > M
    t.limbs[P] = L;
  }
  return t;
}

// Worst-case moduli count for this dtype and K (|S| <= K 2^(2(b + W))).
int wide_planes_max(int bf16, int64_t K) {
  const WideTables t = make_tables();
  const double need = 1.0 + log2(1.0 + 0x1p-5) + log2(static_cast<double>(K > 0 ? K : 1)) +
                      2.0 * (sig_bits(bf16) + wide_spread(bf16)) + 1e-6;
  for (int P = 1; P <= kNumModuliWide; ++P)
    if (t.log2prod[P] > need) return P;
  return -1;
}

// ---------------------------------------------------------------- operands

struct WideOperand {
  const void* X;
  int64_t ld;
  int op;
  int64_t rows, K, Kp;
  int* lo_key;                  // [rows] zeroed: max of (kKeyBias - e) over nonzero elements
  int* hi_key;                  // [rows] zeroed: max of (kKeyBias + e)
  int* nonfinite;               // [rows] zeroed: count of Inf/NaN elements
  unsigned long long* norm;     // [rows] zeroed: bound of sum (X 2^-(b+W))^2, units of 2^-40
  __nv_bfloat16* planes;        // [rows/32][Kp/64][pmax][32][64]
  int pmax;                     // planes' stride (the worst-case count)
  const int* use;               // [rows/64] zeroed: 1 where the 64-row block is in a wide tile
};

// Exponent keys: zero means "no nonzero element", so every per-row statistic
// starts from one memset to zero and is updated with atomicMax.
constexpr int kKeyBias = 1024;                      // e is in [-149, 120]

// Element (r, k) of an operand, and its decode: value = m * 2^e exactly, with
// m < 2^24 (f32) or m < 2^8 (bf16: the significand without its 16 zero bits).
template <int kBf16>
__device__ __forceinline__ uint32_t element_bits(const WideOperand& o, int64_t r, int64_t k) {
  return load_bits<kBf16>(o.X, o.op ? k * o.ld + r : r * o.ld + k);
}

struct WideDecoded {
  int32_t m;
  int32_t e;
  bool nonfinite;
};

template <int kBf16>
__device__ __forceinline__ WideDecoded wide_decode(uint32_t bits) {
  const Decoded d = decode_f32_bits(bits);
  WideDecoded w;
  w.nonfinite = d.nonfinite;
  w.m = kBf16 ? (d.m >> 16) : d.m;            // exact: the low 16 bits are zero
  w.e = kBf16 ? d.e + 16 : d.e;
  return w;
}

// Row r's base (smallest last-bit exponent of a nonzero element), or
// kNoBase if the row is all zero or does not qualify (non-finite elements,
// or a spread beyond the window).
constexpr int kNoBase = 0x7FFFFFFF;
template <int kBf16>
__device__ __forceinline__ int qualifying_base(const WideOperand& o, int64_t r) {
  const int lo = o.lo_key[r], hi = o.hi_key[r];
  if (o.nonfinite[r] != 0 || lo == 0) return kNoBase;
  const int emin = kKeyBias - lo, emax = hi - kKeyBias;
  return emax - emin <= wide_spread(kBf16) ? emin : kNoBase;
}
template <int kBf16>
__device__ __forceinline__ bool row_ok(const WideOperand& o, int64_t r) {
  return o.nonfinite[r] == 0 && (o.lo_key[r] == 0 || qualifying_base<kBf16>(o, r) != kNoBase);
}
// The base of a row the wide GEMM needs: one that qualifies and lies in a
// 64-row block of some wide tile (the routing's flags; a row of no wide tile
// gets no norm and no planes).
template <int kBf16>
__device__ __forceinline__ int row_base(const WideOperand& o, int64_t r) {
  if (o.use != nullptr && o.use[r / kTile] == 0) return kNoBase;
  return qualifying_base<kBf16>(o, r);
}

// Work split of a pass over both operands in one launch: K-contiguous rows,
// one warp per (row, chunk of 2048 k); otherwise one thread per (row, chunk of
// 256 k) with the warp's lanes on neighbouring rows.
constexpr int kRowChunk = 2048;
constexpr int kColChunk = 256;

int64_t pass_blocks(const WideOperand& o) {
  if (o.rows == 0 || o.K == 0) return 0;
  if (o.op == 0) {
    const int64_t warps = o.rows * ((o.K + kRowChunk - 1) / kRowChunk);
    return (warps * 32 + kThreads - 1) / kThreads;
  }
  return ((o.rows + kThreads - 1) / kThreads) * ((o.K + kColChunk - 1) / kColChunk);
}

// Calls f(r, k) for the elements of this thread's share of block `blk` of
// operand o; returns the row and whether this thread reports for it (lane 0
// of the row's warp, or the row's own thread), with warp_reduce applied to
// row-mates' partial results first (K-contiguous layout).
struct PassSlot {
  int64_t r;
  bool reporter;
  bool warp_row;                // the warp shares one row (reduce across lanes)
};

template <typename F>
__device__ __forceinline__ PassSlot for_pass_elements(const WideOperand& o, int64_t blk, F&& f) {
  PassSlot slot{-1, false, false};
  if (o.op == 0) {
    const int64_t chunks = (o.K + kRowChunk - 1) / kRowChunk;
    const int64_t w = (blk * kThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t r = w / chunks;
    if (r >= o.rows) return slot;                   // whole warps
    const int64_t k0 = (w - r * chunks) * kRowChunk;
    const int64_t k1 = min(o.K, k0 + kRowChunk);
    f(r, k0 + lane, k1, int64_t(32));
    slot.r = r;
    slot.reporter = lane == 0;
    slot.warp_row = true;
  } else {
    const int64_t row_blocks = (o.rows + kThreads - 1) / kThreads;
    const int64_t kc = blk / row_blocks;
    const int64_t r = (blk - kc * row_blocks) * kThreads + threadIdx.x;
    if (r >= o.rows) return slot;
    const int64_t k0 = kc * kColChunk, k1 = min(o.K, k0 + kColChunk);
    f(r, k0, k1, int64_t(1));
    slot.r = r;
    slot.reporter = true;
  }
  return slot;
}

// The last block of a launch (all others have finished and published their
// atomics): counter `done` was zeroed before the launch.  No shared memory
// (the flag travels through the barrier's reduction): a kernel that declares
// any does not start beside a running tensor-core GEMM under the default
// carveout.
__device__ __forceinline__ bool last_block(unsigned* done) {
  __threadfence();
  __syncthreads();
  const bool last = __syncthreads_or(threadIdx.x == 0 && atomicAdd(done, 1u) == gridDim.x - 1) != 0;
  if (last) __threadfence();
  return last;
}

struct WideCtl {                 // zeroed with the statistics
  int used;                      // moduli count of the wide GEMM (0: no wide tile)
  int error;                     // the wide GEMM gave up
  unsigned done1, done2;         // block counters of the two passes
  unsigned long long maxA, maxB; // largest row-norm bounds
};

__device__ long long g_route_record[4];              // det_tile_routes

// ---------------------------------------------------------------- pass 1
//
// Per row: exponent keys of its nonzero elements and the count of non-finite
// ones.  The launch's last block then routes: every 64-row block of A and
// 64-column block of C qualifies when all its rows do; each general tile goes
// to the wide list if both its blocks qualify, else it stays with the general
// kernel.  With no general tile nothing runs (and the counts stay zero).
template <int kBf16>
__global__ void __launch_bounds__(kThreads) wide_stats_kernel(WideOperand a, WideOperand b,
                                                              int64_t blocks_a, int64_t blocks_all,
                                                              const int* general,
                                                              int* block_ok, int* wide, int* rest,
                                                              WideCtl* ctl, int* use, int* gflag,
                                                              int* glist, int gemm_rows) {
  const int64_t tiles_m = (a.rows + kTile - 1) / kTile, tiles_n = (b.rows + kTile - 1) / kTile;
  if (general[0] == 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      g_route_record[0] = tiles_m * tiles_n;
      g_route_record[1] = g_route_record[2] = g_route_record[3] = 0;
    }
    return;
  }
  for (int64_t blk = blockIdx.x; blk < blocks_all; blk += gridDim.x) {
    const bool is_a = blk < blocks_a;
    const WideOperand& o = is_a ? a : b;
    int lo = 0, hi = 0, nf = 0;
    const PassSlot slot = for_pass_elements(o, is_a ? blk : blk - blocks_a,
                                            [&](int64_t r, int64_t k, int64_t k1, int64_t step) {
      for (; k < k1; k += step) {
        const WideDecoded d = wide_decode<kBf16>(element_bits<kBf16>(o, r, k));
        nf += d.nonfinite ? 1 : 0;
        if (d.m != 0) {
          lo = max(lo, kKeyBias - d.e);
          hi = max(hi, kKeyBias + d.e);
        }
      }
    });
    if (slot.warp_row) {
      lo = __reduce_max_sync(0xFFFFFFFFu, lo);
      hi = __reduce_max_sync(0xFFFFFFFFu, hi);
      nf = __reduce_add_sync(0xFFFFFFFFu, nf);
    }
    if (slot.reporter) {
      if (lo != 0) atomicMax(o.lo_key + slot.r, lo);
      if (hi != 0) atomicMax(o.hi_key + slot.r, hi);
      if (nf != 0) atomicAdd(o.nonfinite + slot.r, nf);
    }
  }
  if (!last_block(&ctl->done1)) return;
  // the last block: block flags, one warp per 64-row / 64-column block
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int64_t w = wid; w < tiles_m + tiles_n; w += kThreads / 32) {
    const bool blk_a = w < tiles_m;
    const WideOperand& q = blk_a ? a : b;
    const int64_t base = (blk_a ? w : w - tiles_m) * kTile;
    bool ok = true;
#pragma unroll
    for (int h = 0; h < kTile / 32; ++h) {
      const int64_t r = base + lane + 32 * h;
      if (r < q.rows) ok = ok && row_ok<kBf16>(q, r);
    }
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (lane == 0) block_ok[w] = ok ? 1 : 0;
  }
  __syncthreads();
  const int64_t n = general[0];
  for (int64_t i = threadIdx.x; i < n; i += kThreads) {
    const int t = general[1 + i];
    const int64_t tm = t / tiles_n, tn = t - (t / tiles_n) * tiles_n;
    if (block_ok[tm] && block_ok[tiles_m + tn]) wide[1 + atomicAdd(wide, 1)] = t;
    else rest[1 + atomicAdd(rest, 1)] = t;
  }
  __syncthreads();
  // what the wide GEMM needs: the 64-row blocks of A and of B that some wide
  // tile holds (their rows get norms and planes), and the GEMM's own output
  // tiles (gemm_rows x 256) holding a wide tile, listed once each
  const int64_t gemm_tiles_n = (b.rows + 255) / 256;
  const int64_t nw = wide[0];
  for (int64_t i = threadIdx.x; i < nw; i += kThreads) {
    const int t = wide[1 + i];
    const int64_t tm = t / tiles_n, tn = t - (t / tiles_n) * tiles_n;
    use[tm] = 1;
    use[tiles_m + tn] = 1;
    const int64_t gt = (tm * kTile / gemm_rows) * gemm_tiles_n + (tn * kTile) / 256;
    if (atomicExch(gflag + gt, 1) == 0) glist[1 + atomicAdd(glist, 1)] = static_cast<int>(gt);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    g_route_record[0] = tiles_m * tiles_n;
    g_route_record[1] = n;
    g_route_record[2] = wide[0];
    g_route_record[3] = rest[0];
  }
}

// ---------------------------------------------------------------- pass 2
//
// Row norms.  f = X 2^-(b + W) = m 2^(e - base - b - W) is exact (its lowest
// bit is at least 2^-132) and below 1; each thread sums f^2 rounding upwards,
// the warp adds upwards, and the sum, scaled by 2^40 and converted upwards,
// is added to the row's integer bound, never less than the exact sum of
// squares.  The last block then takes the moduli count: with a = max normA,
// b = max normB (units of 2^-40), every S of a wide tile has |S| <= sqrt(a b)
// 2^-40 2^(2(b+W)), and the count is the fewest P whose product exceeds
// 2 (1 + 2^-5) times that (in double, with a margin of 10^-6 bits, far above
// its rounding).  With no wide tile nothing runs (the count stays 0).
template <int kBf16>
__device__ __forceinline__ float scaled_f(int32_t m, int sh) {
  // m * 2^sh with sh in [-(b+W), 0]: two exact scalings by normal powers of two
  return __fmul_rn(__fmul_rn(static_cast<float>(m), 0x1p-64f), __int_as_float((sh + 64 + 127) << 23));
}

__device__ unsigned long long max_norm(const unsigned long long* v, int64_t n) {
  unsigned long long m = 0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) m = max(m, __ldcg(v + i));
#pragma unroll
  for (int s = 16; s >= 1; s /= 2) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, s));
  return m;
}

template <int kBf16>
__global__ void __launch_bounds__(kThreads) wide_norm_kernel(WideOperand a, WideOperand b,
                                                             int64_t blocks_a, int64_t blocks_all,
                                                             const int* wide,
                                                             int pmax, WideCtl* ctl, WideTables t) {
  if (wide[0] == 0) return;
  constexpr int kShift = sig_bits(kBf16) + wide_spread(kBf16);
  for (int64_t blk = blockIdx.x; blk < blocks_all; blk += gridDim.x) {
    const bool is_a = blk < blocks_a;
    const WideOperand& o = is_a ? a : b;
    float sum = 0.0f;
    const PassSlot slot = for_pass_elements(o, is_a ? blk : blk - blocks_a,
                                            [&](int64_t r, int64_t k, int64_t k1, int64_t step) {
      const int base = row_base<kBf16>(o, r);
      if (base == kNoBase) return;                 // zero, or not a wide row: adds nothing
      for (; k < k1; k += step) {
        const WideDecoded d = wide_decode<kBf16>(element_bits<kBf16>(o, r, k));
        if (d.m != 0) {
          const float f = scaled_f<kBf16>(d.m, d.e - base - kShift);
          sum = __fmaf_ru(f, f, sum);
        }
      }
    });
    if (slot.warp_row) {
#pragma unroll
      for (int s = 16; s >= 1; s /= 2) sum = __fadd_ru(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, s));
    }
    if (slot.reporter && sum > 0.0f)
      atomicAdd(o.norm + slot.r, __float2ull_ru(__fmul_ru(sum, 0x1p40f)));
  }
  if (!last_block(&ctl->done2)) return;
  const unsigned long long ma = max_norm(a.norm, a.rows), mb = max_norm(b.norm, b.rows);
  if ((threadIdx.x & 31) == 0) {
    atomicMax(&ctl->maxA, ma);
    atomicMax(&ctl->maxB, mb);
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  const double na = static_cast<double>(atomicAdd(&ctl->maxA, 0ull));
  const double nb = static_cast<double>(atomicAdd(&ctl->maxB, 0ull));
  int P = pmax;
  if (na > 0.0 && nb > 0.0) {
    const double need = 1.0 + log2(1.0 + 0x1p-5) + 0.5 * (log2(na) + log2(nb)) - kNormUnitBits +
                        2.0 * kShift + 1e-6;
    for (int q = 1; q < pmax; ++q)
      if (t.log2prod[q] > need) {
        P = q;
        break;
      }
  } else {
    P = 1;                                        // every product is zero
  }
  ctl->used = P;
}

// ---------------------------------------------------------------- pass 3: residue planes
//
// Persistent over the (32-row group, 64-k stage) tiles of both operands (A's
// first), staged through shared memory (either layout).  Each element of a
// qualifying row with m != 0 is X = m 2^s, s = e - base in [0, W]: its residue
// modulo p is (m mod p) (2^s mod p) mod p, two exact binary32 reductions
// (near_mod_f32: |m mod p| <= 131, |(m mod p)(2^s mod p)| < 2^15, then
// |r| <= (p - 1)/2, or 128 for p = 2^8), the powers of two from a table built
// per block.  Other elements (zero, padding, rows that do not qualify) give
// zero residues.  Only the planes of the chosen count are written; with no
// wide tile nothing runs.
constexpr int kTileRows = 32;
constexpr int kTileK = 64;
constexpr int kMaxShift = 124;                     // wide_spread(bf16)

template <int kBf16>
__global__ void __launch_bounds__(kThreads) wide_planes_kernel(WideOperand a, WideOperand b,
                                                               const WideCtl* ctl) {
  const int P = ctl->used;
  if (P <= 0) return;
  // 18.7 KB of shared memory in all (the powers of two as bf16, exact for
  // |v| <= 256), so that the launch fits beside a running tensor-core GEMM
  // and, with no wide tile, returns there at once
  __shared__ uint32_t tile[kTileRows][kTileK + 1];
  __shared__ int tile_base[kTileRows];
  __shared__ float mod_p[kNumModuliWide], mod_inv[kNumModuliWide];
  __shared__ uint16_t pow2[kNumModuliWide][kMaxShift + 1];
  constexpr int kW = wide_spread(kBf16);
  const int tid = threadIdx.x;
  if (tid < P) {
    const int p = modulus(tid);
    mod_p[tid] = static_cast<float>(p);
    mod_inv[tid] = 1.0f / static_cast<float>(p);
    int v = 1 % p;
    for (int s = 0; s <= kW; ++s) {                 // 2^s mod p, balanced
      const float f = static_cast<float>(v > p / 2 ? v - p : v);
      pow2[tid][s] = static_cast<uint16_t>(__float_as_uint(f) >> 16);   // exact in bf16
      v = (2 * v) % p;
    }
  }
  const int64_t nkb = a.Kp / kStageK;
  const int64_t groups_a = (a.rows + kTileRows - 1) / kTileRows;
  const int64_t groups = groups_a + (b.rows + kTileRows - 1) / kTileRows;
  for (int64_t tix = blockIdx.x; tix < groups * nkb; tix += gridDim.x) {
    const int64_t gg = tix / nkb, kb = tix - (tix / nkb) * nkb;
    const bool is_a = gg < groups_a;
    const WideOperand& o = is_a ? a : b;
    const int64_t g = is_a ? gg : gg - groups_a;
    const int64_t r0 = g * kTileRows, k0 = kb * kTileK;
    if (o.use != nullptr && o.use[r0 / kTile] == 0) continue;   // no wide tile holds these rows
    __syncthreads();                                // tables ready / previous tile done
#pragma unroll
    for (int u = 0; u < kTileRows * kTileK / kThreads; ++u) {
      const int idx = tid + u * kThreads;
      const int r = o.op ? (idx & 31) : (idx >> 6);
      const int k = o.op ? (idx >> 5) : (idx & 63);
      const int64_t gr = r0 + r, gk = k0 + k;
      tile[r][k] = (gr < o.rows && gk < o.K) ? element_bits<kBf16>(o, gr, gk) : 0u;
    }
    if (tid < kTileRows) {
      const int64_t gr = r0 + tid;
      tile_base[tid] = gr < o.rows ? row_base<kBf16>(o, gr) : kNoBase;
    }
    __syncthreads();
#pragma unroll 1
    for (int u = 0; u < kTileRows * kTileK / (2 * kThreads); ++u) {
      const int idx = tid + u * kThreads;
      const int r = idx >> 5, kk = (idx & 31) * 2;
      const int base = tile_base[r];
      float mf[2];
      int sh[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const WideDecoded d = wide_decode<kBf16>(tile[r][kk + h]);
        const bool live = base != kNoBase && d.m != 0;
        mf[h] = live ? static_cast<float>(d.m) : 0.0f;           // exact: |m| < 2^24
        sh[h] = live ? d.e - base : 0;                           // in [0, W]
      }
      uint32_t* dst = reinterpret_cast<uint32_t*>(
          o.planes + (g * nkb + kb) * int64_t(o.pmax) * kPlaneRows * kStageK + r * kStageK + kk);
      for (int q = 0; q < P; ++q) {
        const float p = mod_p[q], inv = mod_inv[q];
        float res[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float r1 = near_mod_f32(mf[h], p, inv);
          const float t = __uint_as_float(static_cast<uint32_t>(pow2[q][sh[h]]) << 16);
          res[h] = near_mod_f32(__fmul_rn(r1, t), p, inv);
        }
        dst[q * (kPlaneRows * kStageK / 2)] =
            __byte_perm(__float_as_uint(res[0]), __float_as_uint(res[1]), 0x7632);
      }
    }
  }
}

// ---------------------------------------------------------------- W6: reconstruction
//
// One block per wide tile at a time (persistent).  The block first builds the
// CRT constants of the chosen count P in shared memory:
//   c_i = (M / p_i)^-1 mod p_i (balanced), C_i = (M / p_i) c_i mod 2^(32 L)
//   as signed 32-bit limbs, -M likewise, W_i = round(2^18 c_i / p_i).
// Per output: S' = sum_i r_i C_i (64-bit limb sums, exact), Q = sum_i r_i W_i,
// q = round(Q / 2^18); since |S/M| <= 1/(2 (1 + 2^-5)) and |Q/2^18 - S'/M|
// <= 40 * 128 * 2^-19 < 0.0098 < 1/2 - 0.4849, q is the integer nearest S'/M
// and S = S' - q M (mod 2^(32 L), which holds it: |S| < M/2 < 2^(32L - 1)).
// Then S 2^(baseA + baseB) as canonical digits: rounded once or written.
constexpr int kOutRows = 64 / (kThreads / 64);      // 16 rows of a tile per thread

struct WideRecon {
  const int8_t* res;              // [pmax][M][N]
  int64_t res_plane;
  const int* wide;                // count, then 64x64 tile indices
  const WideCtl* ctl;             // the moduli count, and the GEMM's error flag
  const int* loA;                 // exponent keys of the rows' smallest elements
  const int* loB;
};

__device__ __forceinline__ void build_constants(int P, int L, int32_t (*C)[12], int32_t* Wt,
                                                int32_t* negM) {
  // thread i < P: C_i and W_i; thread P: -M
  const int i = threadIdx.x;
  if (i > P) return;
  uint32_t w[kMaxLimbs + 1];
#pragma unroll
  for (int l = 0; l <= kMaxLimbs; ++l) w[l] = l == 0 ? 1u : 0u;
  int rm = 1;                                      // (M / p_i) mod p_i
  const int pi = i < P ? modulus(i) : 1;
  for (int j = 0; j < P; ++j) {
    if (j == i) continue;
    const uint32_t pj = static_cast<uint32_t>(modulus(j));
    uint64_t carry = 0;
#pragma unroll
    for (int l = 0; l <= kMaxLimbs; ++l) {
      const uint64_t v = static_cast<uint64_t>(w[l]) * pj + carry;
      w[l] = static_cast<uint32_t>(v);
      carry = v >> 32;
    }
    if (i < P) rm = (rm * (static_cast<int>(pj) % pi)) % pi;
  }
  long long factor = -1;                            // thread P: -M
  if (i < P) {
    int c = 0;
    for (int x = 1; x < pi; ++x)
      if ((rm * x) % pi == 1) {
        c = x;
        break;
      }
    if (pi == 1) c = 0;
    factor = c > (pi - 1) / 2 ? c - pi : c;        // balanced
    // round(2^18 c / p) exactly, in integers
    const long long num = factor * (1ll << (kWeightBits + 1)) + pi;
    const long long den = 2ll * pi;
    Wt[i] = static_cast<int32_t>(num >= 0 ? num / den : -((-num + den - 1) / den));
  }
  // w * factor modulo 2^(32 (kMaxLimbs+1)), two's complement
  const bool neg = factor < 0;
  const uint64_t f = static_cast<uint64_t>(neg ? -factor : factor);
  uint64_t carry = 0;
#pragma unroll
  for (int l = 0; l <= kMaxLimbs; ++l) {
    const uint64_t v = static_cast<uint64_t>(w[l]) * f + carry;
    w[l] = static_cast<uint32_t>(v);
    carry = v >> 32;
  }
  if (neg) {
    uint64_t c = 1;
#pragma unroll
    for (int l = 0; l <= kMaxLimbs; ++l) {
      const uint64_t v = static_cast<uint64_t>(~w[l]) + c;
      w[l] = static_cast<uint32_t>(v);
      c = v >> 32;
    }
  }
  // signed limbs in [-2^31, 2^31): the value mod 2^(32 L) is unchanged
  int64_t borrow = 0;
  int32_t out[12];
#pragma unroll
  for (int l = 0; l < 12; ++l) {
    int64_t v = (l <= kMaxLimbs ? static_cast<int64_t>(w[l]) : 0) + borrow;
    borrow = 0;
    if (v >= (int64_t(1) << 31)) {
      v -= int64_t(1) << 32;
      borrow = 1;
    }
    out[l] = static_cast<int32_t>(v);
  }
  (void)L;
  if (i < P) {
#pragma unroll
    for (int l = 0; l < 12; ++l) C[i][l] = out[l];
  } else {
#pragma unroll
    for (int l = 0; l < 12; ++l) negM[l] = out[l];
  }
}

// The exact value S 2^E (S in L signed limbs) as canonical digits: 17 words
// and a signed top (bit 0 of the digits weighs 2^-298, E >= -298).
template <int L>
__device__ __forceinline__ void place_digits(const uint32_t (&x)[L], int E, uint32_t (&w)[kDigits - 1],
                                             int64_t& top) {
  const int off = E + kLsbBias;
  const int j0 = off >> 5, sh = off & 31;
  const uint32_t sx = static_cast<uint32_t>(static_cast<int32_t>(x[L - 1]) >> 31);
  uint32_t y[L + 1];
  y[0] = x[0] << sh;
#pragma unroll
  for (int i = 1; i < L; ++i) y[i] = __funnelshift_l(x[i - 1], x[i], sh);
  y[L] = __funnelshift_l(x[L - 1], sx, sh);
  uint32_t d17 = 0;
#pragma unroll
  for (int j = 0; j < kDigits; ++j) {
    const int k = j - j0;
    uint32_t v = k < 0 ? 0u : sx;
#pragma unroll
    for (int i = 0; i <= L; ++i) v = (k == i) ? y[i] : v;
    if (j < kDigits - 1) w[j] = v;
    else d17 = v;
  }
  top = static_cast<int64_t>(static_cast<int32_t>(d17));
}

// RNE_f32(S 2^E) from S's limbs: the leading 64 bits of |S|, with every bit
// below them ORed into bit 0 (a sticky bit far below the rounding position),
// round to binary32 exactly as |S| does; the scaling by a power of two is an
// exponent add.  Returns false (the caller takes the digit route) where the
// result is subnormal, zero or infinite.
template <int L>
__device__ __forceinline__ bool round_limbs_fast(const uint32_t (&x)[L], int E, uint32_t& bits) {
  const bool neg = static_cast<int32_t>(x[L - 1]) < 0;
  uint32_t a[L];
  uint32_t carry = neg ? 1u : 0u;
#pragma unroll
  for (int l = 0; l < L; ++l) {                   // |S| (two's complement negation if negative)
    const uint32_t v = neg ? ~x[l] : x[l];
    a[l] = v + carry;
    carry = (carry != 0u && a[l] == 0u) ? 1u : 0u;
  }
  int top = -1;
#pragma unroll
  for (int l = 0; l < L; ++l) top = a[l] != 0u ? l : top;
  if (top < 0) {                                  // exact zero -> +0
    bits = 0u;
    return true;
  }
  // the three words from the leading one down, and the OR of the rest
  uint32_t w2 = 0, w1 = 0, w0 = 0, rest = 0;
#pragma unroll
  for (int l = 0; l < L; ++l) {
    if (l == top) w2 = a[l];
    if (l == top - 1) w1 = a[l];
    if (l == top - 2) w0 = a[l];
    if (l < top - 2) rest |= a[l];
  }
  const int lz = __clz(w2);                       // 0 .. 31
  const uint64_t hi64 = (static_cast<uint64_t>(w2) << 32) | w1;
  uint64_t t = lz ? (hi64 << lz) | (w0 >> (32 - lz)) : hi64;
  const uint32_t below = lz ? (w0 << lz) : w0;
  t |= (below | rest) != 0u ? 1u : 0u;
  const uint32_t f = f32_bits_of_top(t);          // |S| 2^-(32 top + 32 - lz - 64), rounded
  const int shift = E + 32 * top + 32 - lz - 64;
  const int ef = static_cast<int>(f >> 23) + shift;   // biased exponent of the result
  if (ef < 1 || ef > 254) return false;
  bits = (neg ? 0x80000000u : 0u) | (f + (static_cast<uint32_t>(shift) << 23));
  return true;
}

// The digit route of one output: rare for det_gemm (subnormal, zero or
// infinite results), kept out of line so the main loop keeps its registers.
template <int L>
__device__ __noinline__ uint32_t round_limbs_exact(const uint32_t (&x)[L], int E) {
  uint32_t w[kDigits - 1];
  int64_t top;
  place_digits<L>(x, E, w, top);
  return round_to_f32_bits(w, top);
}

template <int L>
__device__ void wide_recon_body(const GemmArgs& g, const WideRecon& wr, int P,
                                const int32_t (*C)[12], const int32_t* Wt, const int32_t* negM) {
  const int64_t MN = g.M * g.N;
  const int64_t tiles_n = (g.N + kTile - 1) / kTile;
  const bool failed = wr.ctl->error != 0;
  const int64_t ntiles = wr.wide[0];
  const int tid = threadIdx.x;
  for (int64_t ti = blockIdx.x; ti < ntiles; ti += gridDim.x) {
    const int t = wr.wide[1 + ti];
    const int64_t m0 = (t / tiles_n) * kTile, n0 = (t - (t / tiles_n) * tiles_n) * kTile;
    const int64_t n = n0 + (tid & 63);
    if (n >= g.N) continue;
    // the row's base (an all-zero row or column has none: its S is zero, and
    // any E places it)
    const int bB = wr.loB[n] != 0 ? kKeyBias - wr.loB[n] : 0;
    for (int i = 0; i < kOutRows; i += 2) {
      int64_t m[2];
      bool live[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        m[h] = m0 + (tid >> 6) + 4 * (i + h);
        live[h] = m[h] < g.M;
      }
      if (!live[0]) break;
      int64_t acc[2][L];
      int32_t Q[2] = {0, 0};
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int l = 0; l < L; ++l) acc[h][l] = 0;
      for (int q = 0; q < P; ++q) {
        int32_t r[2];
#pragma unroll
        for (int h = 0; h < 2; ++h)
          r[h] = live[h] ? static_cast<int32_t>(wr.res[q * wr.res_plane + m[h] * g.N + n]) : 0;
        const int32_t wq = Wt[q];
        int32_t c[12];                              // the limbs, 16 bytes at a time
#pragma unroll
        for (int l4 = 0; l4 < (L + 3) / 4; ++l4) {
          const int4 v = reinterpret_cast<const int4*>(C[q])[l4];
          c[4 * l4] = v.x;
          c[4 * l4 + 1] = v.y;
          c[4 * l4 + 2] = v.z;
          c[4 * l4 + 3] = v.w;
        }
#pragma unroll
        for (int l = 0; l < L; ++l) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
            asm("mad.wide.s32 %0, %1, %2, %0;" : "+l"(acc[h][l]) : "r"(r[h]), "r"(c[l]));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) Q[h] += r[h] * wq;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!live[h]) continue;
        const int32_t qq = (Q[h] + (1 << (kWeightBits - 1))) >> kWeightBits;
#pragma unroll
        for (int l = 0; l < L; ++l) acc[h][l] += static_cast<int64_t>(qq) * negM[l];
        // carry into 32-bit limbs: S modulo 2^(32 L), two's complement
        uint32_t x[L];
        int64_t carry = 0;
#pragma unroll
        for (int l = 0; l < L; ++l) {
          const int64_t v = acc[h][l] + carry;
          x[l] = static_cast<uint32_t>(v);
          carry = v >> 32;
        }
        const int bA = wr.loA[m[h]] != 0 ? kKeyBias - wr.loA[m[h]] : 0;
        const int E = bA + bB;
        if (g.P == nullptr) {
          uint32_t bits;
          if (failed) {
            bits = kNanBits;
          } else if (!round_limbs_fast<L>(x, E, bits)) {   // subnormal, zero or infinite
            bits = round_limbs_exact<L>(x, E);
          }
          reinterpret_cast<uint32_t*>(g.C)[m[h] * g.ldc + n] = bits;
          continue;
        }
        uint32_t w[kDigits - 1];
        int64_t top;
        place_digits<L>(x, E, w, top);
        {
          int64_t* out = g.P + m[h] * g.N + n;
#pragma unroll
          for (int j = 0; j < kDigits - 1; ++j) out[j * MN] = failed ? 0 : static_cast<int64_t>(w[j]);
          out[(kDigits - 1) * MN] = failed ? 0 : top;
          out[kDigits * MN] = g.K;
          out[(kDigits + 1) * MN] = failed ? 1 : 0;
        }
      }
    }
  }
  (void)tiles_n;
}

__global__ void __launch_bounds__(kThreads) wide_recon_kernel(GemmArgs g, WideRecon wr, WideTables t) {
  const int P = wr.ctl->used;
  if (P <= 0 || wr.wide[0] == 0) return;
  __shared__ __align__(16) int32_t C[kNumModuliWide][12];
  __shared__ int32_t Wt[kNumModuliWide];
  __shared__ int32_t negM[12];
  const int L = t.limbs[P];
  build_constants(P, L, C, Wt, negM);
  __syncthreads();
  switch (L) {
    case 1: case 2: case 3: case 4: wide_recon_body<4>(g, wr, P, C, Wt, negM); break;
    case 5: wide_recon_body<5>(g, wr, P, C, Wt, negM); break;
    case 6: wide_recon_body<6>(g, wr, P, C, Wt, negM); break;
    case 7: wide_recon_body<7>(g, wr, P, C, Wt, negM); break;
    case 8: wide_recon_body<8>(g, wr, P, C, Wt, negM); break;
    case 9: wide_recon_body<9>(g, wr, P, C, Wt, negM); break;
    default: wide_recon_body<10>(g, wr, P, C, Wt, negM); break;
  }
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Zeroes n 16-byte words: small blocks with few registers, so that the launch
// fits beside a running tensor-core CTA (a driver memset may not).
__global__ void __launch_bounds__(kThreads) zero_kernel(uint4* p, int64_t n) {
  for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < n; i += int64_t(gridDim.x) * kThreads)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

int sm_count() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

}  // namespace

int route_record(long long* out) {
  long long rec[4];
  if (cudaMemcpyFromSymbol(rec, g_route_record, sizeof(rec)) != cudaSuccess) return -1;
  for (int i = 0; i < 4; ++i) out[i] = rec[i];
  return 0;
}

// The general tiles of a residue-path call: the wide path where the rows
// qualify, the general kernel for the rest.  wide_prepare enqueues, on
// `stream` after the routing (route and general list in s), the row
// statistics, routing, norms and planes, and records ev_planes;
// wide_finish enqueues the wide tensor-core GEMM, the wide reconstruction and
// the general kernel on `tail` after ev_planes.  With no general tile every
// one of these kernels returns at once.
cudaError_t wide_prepare(const GemmArgs& g, const Scratch& s, cudaStream_t stream,
                         cudaEvent_t ev_planes, WidePlan* plan) {
  WidePlan& w = *plan;
  w = WidePlan{};
  const int bf16 = g.bf16;
  const int pmax = wide_planes_max(bf16, g.K);
  const int64_t Kp = (g.K + kStageK - 1) / kStageK * kStageK;
  const int64_t tiles_m = (g.M + kTile - 1) / kTile, tiles_n = (g.N + kTile - 1) / kTile;
  const int64_t tiles = tiles_m * tiles_n;
  w.general = s.general;
  // scratch: per-row statistics, routing lists, planes and residues; the
  // planes and residues are sized for the worst-case count
  const size_t rows = static_cast<size_t>(g.M + g.N);
  const size_t planes_bytes = 2 * size_t(pmax) * (size_t(plane_rows(g.M)) + size_t(plane_rows(g.N))) *
                              size_t(Kp);
  const size_t res_bytes = size_t(pmax) * size_t(g.M) * size_t(g.N);
  // too large a problem for the worst-case scratch: the general kernel alone
  if (pmax < 0 || planes_bytes + res_bytes > (size_t(16) << 30) ||
      (g.M + 31) / 32 > 65535 || (g.N + 31) / 32 > 65535) {
    w.active = false;
    return cudaEventRecord(ev_planes, stream);
  }
  w.active = true;
  size_t off = 0;                    // zeroed together: statistics, block flags, lists, control
  const size_t o_lo = off;           off = align_up(off + 4 * rows, 256);
  const size_t o_hi = off;           off = align_up(off + 4 * rows, 256);
  const size_t o_nf = off;           off = align_up(off + 4 * rows, 256);
  const size_t o_norm = off;         off = align_up(off + 8 * rows, 256);
  const size_t o_blk = off;          off = align_up(off + 4 * size_t(tiles_m + tiles_n), 256);
  const size_t o_wide = off;         off = align_up(off + 4 * size_t(tiles + 1), 256);
  const size_t o_rest = off;         off = align_up(off + 4 * size_t(tiles + 1), 256);
  const size_t o_ctl = off;          off = align_up(off + sizeof(WideCtl), 256);
  // the wide GEMM's tiles: gemm_rows x 256 (CTA pairs, or one CTA for M <= 128)
  const int gemm_rows = g.M > 128 ? 256 : 128;
  const int64_t gemm_tiles = ((g.M + gemm_rows - 1) / gemm_rows) * ((g.N + 255) / 256);
  const size_t o_use = off;          off = align_up(off + 4 * size_t(tiles_m + tiles_n), 256);
  const size_t o_gflag = off;        off = align_up(off + 4 * size_t(gemm_tiles), 256);
  const size_t o_glist = off;        off = align_up(off + 4 * size_t(gemm_tiles + 1), 256);
  const size_t zero_bytes = off;
  off = align_up(off, 1024);
  const size_t o_pa = off;           off = align_up(off + 2 * size_t(pmax) * plane_rows(g.M) * Kp, 1024);
  const size_t o_pb = off;           off = align_up(off + 2 * size_t(pmax) * plane_rows(g.N) * Kp, 1024);
  const size_t o_res = off;          off = align_up(off + res_bytes, 1024);
  cudaError_t e = pool_alloc(&w.mem, off, stream);
  if (e != cudaSuccess) return e;
  char* base = static_cast<char*>(w.mem);
  int* lo = reinterpret_cast<int*>(base + o_lo);
  int* hi = reinterpret_cast<int*>(base + o_hi);
  int* nf = reinterpret_cast<int*>(base + o_nf);
  unsigned long long* norm = reinterpret_cast<unsigned long long*>(base + o_norm);
  int* blk = reinterpret_cast<int*>(base + o_blk);
  w.wide = reinterpret_cast<int*>(base + o_wide);
  w.rest = reinterpret_cast<int*>(base + o_rest);
  w.ctl = base + o_ctl;
  WideCtl* ctl = reinterpret_cast<WideCtl*>(w.ctl);
  w.planesA = reinterpret_cast<__nv_bfloat16*>(base + o_pa);
  w.planesB = reinterpret_cast<__nv_bfloat16*>(base + o_pb);
  w.res = reinterpret_cast<int8_t*>(base + o_res);
  w.loA = lo;
  w.loB = lo + g.M;
  w.pmax = pmax;
  w.Kp = Kp;

  int* use = reinterpret_cast<int*>(base + o_use);
  int* gflag = reinterpret_cast<int*>(base + o_gflag);
  w.glist = reinterpret_cast<int*>(base + o_glist);
  WideOperand oa{g.A, g.lda, g.opA, g.M, g.K, Kp, lo, hi, nf, norm, w.planesA, pmax, use};
  WideOperand ob{g.B, g.ldb, g.opB, g.N, g.K, Kp, lo + g.M, hi + g.M, nf + g.M, norm + g.M,
                 w.planesB, pmax, use + tiles_m};
  const WideTables tables = make_tables();
  const int sms = sm_count();
  // the kernels with shared memory prefer the largest carveout, so that they
  // can start on an SM beside a running tensor-core CTA
  static PerDeviceOnce carveout;
  carveout.run([](int) {
    const int pref = cudaSharedmemCarveoutMaxShared;
    cudaFuncSetAttribute(wide_planes_kernel<0>, cudaFuncAttributePreferredSharedMemoryCarveout, pref);
    cudaFuncSetAttribute(wide_planes_kernel<1>, cudaFuncAttributePreferredSharedMemoryCarveout, pref);
    cudaFuncSetAttribute(wide_recon_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, pref);
    cudaGetLastError();                            // a preference only: never the caller's error
    return cudaSuccess;
  });
  const int64_t ba = pass_blocks(oa), bb = pass_blocks(ob);
  {
    StageScope t(kStageWideStats, stream);
    if (e == cudaSuccess) {
      const int64_t words = static_cast<int64_t>(zero_bytes / 16);     // a multiple of 256 bytes
      const int64_t grid = (words + 8 * kThreads - 1) / (8 * kThreads);
      zero_kernel<<<static_cast<unsigned>(grid < int64_t(sms) ? grid : int64_t(sms)), kThreads, 0,
                    stream>>>(reinterpret_cast<uint4*>(base), words);
      note_launch();
      e = cudaGetLastError();
    }
    if (e == cudaSuccess && ba + bb > 0) {
      // persistent: at most four blocks per SM walk the passes' blocks
      const int64_t all = ba + bb;
      const unsigned grid = static_cast<unsigned>(all < int64_t(sms) * 4 ? all : int64_t(sms) * 4);
      if (bf16)
        wide_stats_kernel<1><<<grid, kThreads, 0, stream>>>(oa, ob, ba, all, s.general, blk, w.wide,
                                                            w.rest, ctl, use, gflag, w.glist, gemm_rows);
      else
        wide_stats_kernel<0><<<grid, kThreads, 0, stream>>>(oa, ob, ba, all, s.general, blk, w.wide,
                                                            w.rest, ctl, use, gflag, w.glist, gemm_rows);
      if (bf16) wide_norm_kernel<1><<<grid, kThreads, 0, stream>>>(oa, ob, ba, all, w.wide, pmax, ctl, tables);
      else wide_norm_kernel<0><<<grid, kThreads, 0, stream>>>(oa, ob, ba, all, w.wide, pmax, ctl, tables);
      note_launch(2);
      e = cudaGetLastError();
    }
  }
  {
    StageScope t(kStageWidePlanes, stream);
    if (e == cudaSuccess) {
      const int64_t tiles_o = ((g.M + kTileRows - 1) / kTileRows + (g.N + kTileRows - 1) / kTileRows) *
                              (Kp / kStageK);
      const int64_t grid = tiles_o < int64_t(sms) * 4 ? tiles_o : int64_t(sms) * 4;
      if (bf16) wide_planes_kernel<1><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(oa, ob, ctl);
      else wide_planes_kernel<0><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(oa, ob, ctl);
      note_launch();
      e = cudaGetLastError();
    }
  }
  if (e == cudaSuccess) e = cudaEventRecord(ev_planes, stream);
  if (e != cudaSuccess) {                          // nothing will use the scratch
    cudaFreeAsync(w.mem, stream);
    w.mem = nullptr;
    w.active = false;
  }
  return e;
}

cudaError_t wide_finish(const GemmArgs& g, const WidePlan& w, cudaStream_t tail,
                        cudaEvent_t ev_planes) {
  cudaError_t e = cudaStreamWaitEvent(tail, ev_planes, 0);
  if (e != cudaSuccess) return e;
  if (!w.active) {
    StageScope t(kStageGeneral, tail);
    return launch_kulisch(g, w.general, true, tail);
  }
  unsigned* status = nullptr;
  e = device_status_word(&status);
  WideCtl* ctl = reinterpret_cast<WideCtl*>(w.ctl);
  const int64_t tiles = ((g.M + kTile - 1) / kTile) * ((g.N + kTile - 1) / kTile);
  const int sms = sm_count();
  if (e == cudaSuccess) {
    StageScope t(kStageWideGemm, tail);
    // sized for the worst-case count (clusters beyond the work return at
    // once); with no wide tile the count is 0 and every CTA returns at entry
    ResGemmArgs rg{w.planesA, w.planesB, g.M, g.N, w.Kp, w.pmax, w.res, g.M * g.N, &ctl->error,
                   status, &ctl->used, 1, w.pmax};
    rg.tile_list = w.glist;                // only the output tiles holding a wide tile
    e = g.M > 128 ? launch_residue_gemm_pair(rg, tail) : cudaErrorNotSupported;
    if (e == cudaErrorNotSupported) {
      if (g.M > 128) rg.tile_list = nullptr;   // the list names 256-row tiles: every tile instead
      e = launch_residue_gemm(rg, tail);
    }
  }
  if (e == cudaSuccess) {
    StageScope t(kStageWideReconstruct, tail);
    WideRecon wr{w.res, g.M * g.N, w.wide, ctl, w.loA, w.loB};
    const int64_t grid = tiles < int64_t(sms) * 4 ? tiles : int64_t(sms) * 4;
    wide_recon_kernel<<<static_cast<unsigned>(grid > 0 ? grid : 1), kThreads, 0, tail>>>(
        g, wr, make_tables());
    note_launch();
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    StageScope t(kStageGeneral, tail);
    e = launch_kulisch(g, w.rest, true, tail);
  }
  // every user of the scratch is on `tail` (or before ev_planes)
  const cudaError_t f = cudaFreeAsync(w.mem, tail);
  return e != cudaSuccess ? e : f;
}

}  // namespace det
