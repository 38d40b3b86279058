// Residue (CRT) decomposition of the exact GEMM, the CUDA-core halves:
//   residue_kernel      operands -> bf16 residue planes + per-row deep lists
//   reconstruct_*       residues of the shallow dot product -> exact value
//                       (CRT) + deep products -> round once (or digits)
//
// Shallow elements.  For a row r of an operand with largest last-bit
// exponent emax[r], an element m*2^e with e >= emax[r] - 18 is the integer
//     X_int = m * 2^(e - emax[r] + 18)
// times 2^(emax[r] - 18), with |X_int| < 2^42 (f32) or 2^26 (bf16, whose
// significand has 8 bits).  So for an output (m, n) the shallow products sum
// to 2^(emaxA[m] + emaxB[n] - 36) * S with S = sum_k A_int[m,k] * B_int[n,k],
// an exact integer dot product, |S| <= ||A_int[m,:]|| ||B_int[n,:]|| (Cauchy-
// Schwarz) <= K * 2^84.  S is computed modulo P small odd pairwise-coprime
// moduli (residues in bf16 planes, multiplied on tensor cores with exact fp32
// accumulation) and rebuilt here by the Chinese remainder theorem: the
// moduli's product exceeds 2|S| (1 + 2^-7).  The planes are written for the
// count that the worst case K * 2^84 needs; the residue kernel also sums an
// upper bound of each row's squared norm, and a one-block kernel picks per
// row band the smallest count that the Cauchy-Schwarz bound allows (12 rather
// than 13 for N(0,1) data at K = 4096).  The tensor-core GEMM and the
// reconstruction read that count from device memory, so no host round trip
// is needed.  All the small modular arithmetic runs in exact binary32 on the
// FMA pipes.
// Deep elements (more than 18 binades below the row max) and non-finite ones
// are left out of the planes and listed per row; their products are added
// exactly, one by one, during reconstruction.  Together this is the exact sum
// of the products rounded once to fp32, as the det-train page's "Method"
// section defines it; only the order of the exact integer additions differs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "det_arith.cuh"
#include "det_crt.cuh"
#include "det_gemm_internal.cuh"
#include "det_kernels.h"
#include "det_residue.cuh"
#include "tc_ptx.cuh"

#include <atomic>
#include <type_traits>

namespace det {

// The moduli counts most recently chosen per row band (a diagnostic,
// det_moduli_used; concurrent calls overwrite one another's entries).
constexpr int kModuliRecord = 8;
__device__ int g_moduli_record[kModuliRecord];

namespace {

bool rows_layout(const ResidueOperand& o, int bf16) {
  // vector loads: K-contiguous rows whose every row start is 16-byte (f32) or
  // 8-byte (bf16) aligned
  const uintptr_t vec = bf16 ? 8 : 16;
  return o.op == 0 && (reinterpret_cast<uintptr_t>(o.X) % vec) == 0 &&
         (o.ld * (bf16 ? 2 : 4)) % int64_t(vec) == 0 &&
         (o.group_rows <= 0 || (int64_t(o.group_stride) * (bf16 ? 2 : 4)) % int64_t(vec) == 0);
}

constexpr int kThreads = 256;
constexpr int kTileRows = 32;

// A row's deep-element list slot, taken one by one.  Taken this way the
// count saturates a little past the list's capacity (the fused kernel's
// warps that count their deep elements first add them all at once): once a
// row holds more deep elements than its list takes,
// every tile of the row goes to the general tiles, and every reader of the
// count only asks whether it exceeds the capacity (or is nonzero), so further
// increments are skipped.  Without this, data whose elements are nearly all
// deep (exponents spread over hundreds of binades) piled millions of atomic
// increments onto a few hundred counters.  Returns the slot taken, or a value
// past the capacity when none was taken.
__device__ __forceinline__ int take_deep_slot(int* count, int cap) {
  if (__ldcg(count) > cap) return cap + 1;
  return atomicAdd(count, 1);
}

// Whether every row of a block's 32 is past its deep list's capacity: such a
// row is general on every tile (the routing sends each tile holding it to the
// general tiles), so nothing the planes kernels would write for it -- its
// residues, list entries, norm -- is read again; padding rows are read only
// for outputs past M or N.  The two-pass kernels, whose blocks each take one
// 64-k stage of 32 rows, skip such blocks (data whose rows are nearly all
// deep elements, such as exponents spread over hundreds of binades).
__device__ __forceinline__ bool rows_past_capacity(const ResidueOperand& o, int64_t r0) {
  const int64_t gr = r0 + threadIdx.x;
  const int past = threadIdx.x >= kTileRows || gr >= o.rows || __ldcg(o.list_count + gr) > o.cap;
  return __syncthreads_and(past) != 0;
}

constexpr int kTileK = 64;

// Reduction modulo a compile-time modulus (near_mod_f32 states the bounds).
template <int p>
__device__ __forceinline__ float near_mod(float a) {
  constexpr float inv = 1.0f / static_cast<float>(p);
  return near_mod_f32(a, static_cast<float>(p), inv);
}

// A residue, modulo the compile-time modulus p, of the integer x * 2^s given
// x (|x| < 2^24, exact in binary32) and pw = 2^s (s in [0, 18]):
//   r1 = x mod p (|r1| < 131),  u = r1 * 2^s (exact, |u| < 2^26),
//   result = u mod p, with |result| <= 138.
// A zero residue is +0 (x = +0 gives r1 = +0, and pw > 0).
template <int p>
__device__ __forceinline__ float residue_f32(float x, float pw) {
  return near_mod<p>(__fmul_rn(near_mod<p>(x), pw));
}

// bf16 pair of two small integers held exactly in binary32: the top halves of
// their bit patterns (the low halves are zero).
__device__ __forceinline__ uint32_t bf16_pair(float lo, float hi) {
  return __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);
}

// Plane i of an element pair sits one 32 x 64 block (4 KB, 1024 bf16 pairs)
// after plane i - 1.
template <int i, int P>
__device__ __forceinline__ void write_residue_pairs(uint32_t* dst, float x0, float pw0, float x1,
                                                    float pw1) {
  if constexpr (i < P) {
    constexpr int p = modulus(i);
    dst[i * (kPlaneRows * kStageK / 2)] = bf16_pair(residue_f32<p>(x0, pw0), residue_f32<p>(x1, pw1));
    write_residue_pairs<i + 1, P>(dst, x0, pw0, x1, pw1);
  }
}

// Adds the shallow elements' X_int^2 / 2^norm_shift held by this thread to
// its row's norm bound.  The kLanes neighbouring lanes that share the row
// reduce first (every step rounds to nearest: at most 8 roundings of
// positive values, relative error below 2^-20); one lane then adds the sum
// scaled by 1 + 2^-19 and converted upwards, never less than the exact sum.
// Zero, deep and padding elements carry x = 0.
template <int kBf16, int kLanes, int kN>
__device__ __forceinline__ void add_row_norm(const ResidueOperand& o, int64_t gr, const float (&x)[kN],
                                             const float (&pw)[kN]) {
  constexpr float kHalfShift = kBf16 ? 0x1p-8f : 0x1p-26f;      // 2^(-norm_shift / 2)
  static_assert(norm_shift(kBf16) == (kBf16 ? 16 : 52), "kHalfShift squared is 2^-norm_shift");
  float sum = 0.0f;
#pragma unroll
  for (int h = 0; h < kN; ++h) {
    const float f = __fmul_rn(__fmul_rn(x[h], pw[h]), kHalfShift);   // exact
    sum = __fmaf_rn(f, f, sum);
  }
#pragma unroll
  for (int w = kLanes / 2; w >= 1; w /= 2) sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, w));
  if ((threadIdx.x & (kLanes - 1)) == 0 && gr < o.rows && sum > 0.0f && o.norm != nullptr)
    atomicAdd(o.norm + gr, __float2ull_ru(__fmul_ru(sum, 1.0f + 0x1p-19f)));
}

// One block: one group of 32 rows x one 64-k stage of one operand; each
// thread then handles pairs of neighbouring k, writing the P residues of a
// pair as P 4-byte words 4 KB apart (a warp covers one row's stage: one
// 128-byte line per plane).  Padding rows get zero residues.  Every deep or
// non-finite element is counted (and listed while there is room).
// Two operands may share a launch: blocks with blockIdx.y below `split` take
// o0, the others o1 (row block blockIdx.y - split).
template <int kBf16, int P>
__global__ void __launch_bounds__(kThreads) residue_kernel(ResidueOperand o0, ResidueOperand o1,
                                                           unsigned split) {
  static_assert(kTileK == kStageK && kTileRows == kPlaneRows, "one block covers one plane block");
  __shared__ uint32_t tile[kTileRows][kTileK + 1];
  __shared__ int row_emax[kTileRows];
  const bool second = blockIdx.y >= split;
  const ResidueOperand o = second ? o1 : o0;
  const int64_t by = second ? blockIdx.y - split : blockIdx.y;
  const int tid = threadIdx.x;
  const int64_t r0 = by * kTileRows;
  const int64_t k0 = int64_t(blockIdx.x) * kTileK;
  if (rows_past_capacity(o, r0)) return;
#pragma unroll
  for (int u = 0; u < kTileRows * kTileK / kThreads; ++u) {
    const int idx = tid + u * kThreads;
    const int r = o.op ? (idx & 31) : (idx >> 6);
    const int k = o.op ? (idx >> 5) : (idx & 63);
    const int64_t gr = r0 + r, gk = k0 + k;
    uint32_t bits = 0;
    if (gr < o.rows && gk < o.K) bits = load_bits<kBf16>(o.X, o.op ? gk * o.ld + gr : gr * o.ld + gk);
    tile[r][k] = bits;
  }
  if (tid < kTileRows) {
    const int em = r0 + tid < o.rows ? o.emax[r0 + tid] : 0;
    row_emax[tid] = em == kEmaxEmpty ? 0 : em;
  }
  __syncthreads();
  const int64_t nkb = o.Kp / kStageK;
#pragma unroll 1
  for (int u = 0; u < kTileRows * kTileK / (2 * kThreads); ++u) {
    const int idx = tid + u * kThreads;
    const int r = idx >> 5, kk = (idx & 31) * 2;
    const int64_t gr = r0 + r, gk = k0 + kk;
    const int em = row_emax[r];
    float x[2], pw[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t bits = tile[r][kk + h];
      const Decoded d = decode_f32_bits(bits);
      const int s = d.e - em + kDeepGap;
      const bool deep = d.nonfinite || (d.m != 0 && s < 0);
      // a bf16 significand widened to binary32 carries 16 zero bits: drop them
      // (exactly) so that |X_int| < 2^26; the reconstruction scales back by 2^32
      const int32_t mi = kBf16 ? (d.m >> 16) : d.m;
      x[h] = static_cast<float>(deep ? 0 : mi);                        // exact: |mi| < 2^24
      pw[h] = __int_as_float((deep || d.m == 0 ? 127 : s + 127) << 23);  // 2^s, s in [0, 18]
      if (deep && gk + h < o.K && gr < o.rows) {
        const int slot = take_deep_slot(o.list_count + gr, o.cap);
        if (slot < o.cap) o.list[gr * o.cap + slot] = make_uint2(static_cast<uint32_t>(gk + h), bits);
      }
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>(
        o.planes + (by * nkb + int64_t(blockIdx.x)) * P * kPlaneRows * kStageK +
        r * kStageK + kk);
    write_residue_pairs<0, P>(dst, x[0], pw[0], x[1], pw[1]);
    add_row_norm<kBf16, 32>(o, gr, x, pw);                  // a warp covers the row's stage
  }
}

// Four neighbouring elements' residues: plane i gets one 8-byte word of four
// bf16 values, one 32 x 64 block (4 KB, 512 8-byte words) after plane i - 1.
template <int i, int P>
__device__ __forceinline__ void write_residue_quads(uint2* dst, const float (&x)[4],
                                                    const float (&pw)[4]) {
  if constexpr (i < P) {
    constexpr int p = modulus(i);
    // evict-first: the planes are read back by a later launch, and a later
    // band's are written while a GEMM's own planes need L2
    __stcs(&dst[i * (kPlaneRows * kStageK / 4)],
           make_uint2(bf16_pair(residue_f32<p>(x[0], pw[0]), residue_f32<p>(x[1], pw[1])),
                      bf16_pair(residue_f32<p>(x[2], pw[2]), residue_f32<p>(x[3], pw[3]))));
    write_residue_quads<i + 1, P>(dst, x, pw);
  }
}

// The residue kernel for K-contiguous operands (op 0) whose rows start on a
// vector boundary: no shared-memory staging.  A block covers one group of 32
// rows x one 64-k stage; each thread takes two runs of 4 neighbouring k
// (one 16-byte f32 or 8-byte bf16 load each) and writes each plane as one
// 8-byte word, so a half-warp stores one 128-byte plane row.
template <int kBf16, int P>
__global__ void __launch_bounds__(kThreads) residue_rows_kernel(ResidueOperand o0, ResidueOperand o1,
                                                                unsigned split) {
  const bool second = blockIdx.y >= split;
  const ResidueOperand o = second ? o1 : o0;
  const int64_t by = second ? blockIdx.y - split : blockIdx.y;
  const int tid = threadIdx.x;
  const int64_t r0 = by * kTileRows;
  const int64_t k0 = int64_t(blockIdx.x) * kTileK;
  const int64_t nkb = o.Kp / kStageK;
  if (rows_past_capacity(o, r0)) return;
#pragma unroll 1
  for (int u = 0; u < kTileRows * kTileK / (4 * kThreads); ++u) {
    const int idx = tid + u * kThreads;
    const int r = idx >> 4, kq = (idx & 15) * 4;
    const int64_t gr = r0 + r, gk = k0 + kq;
    uint32_t bits[4] = {0u, 0u, 0u, 0u};
    int em = 0;
    if (gr < o.rows) {
      em = o.emax[gr];
      em = em == kEmaxEmpty ? 0 : em;
      if (gk + 4 <= o.K) {
        if (kBf16) {
          const uint2 v = __ldg(reinterpret_cast<const uint2*>(
              static_cast<const uint16_t*>(o.X) + gr * o.ld + gk));
          bits[0] = v.x << 16;
          bits[1] = v.x & 0xFFFF0000u;
          bits[2] = v.y << 16;
          bits[3] = v.y & 0xFFFF0000u;
        } else {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(
              static_cast<const uint32_t*>(o.X) + gr * o.ld + gk));
          bits[0] = v.x;
          bits[1] = v.y;
          bits[2] = v.z;
          bits[3] = v.w;
        }
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h)
          if (gk + h < o.K) bits[h] = load_bits<kBf16>(o.X, gr * o.ld + gk + h);
      }
    }
    float x[4], pw[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const Decoded d = decode_f32_bits(bits[h]);
      const int s = d.e - em + kDeepGap;
      const bool deep = d.nonfinite || (d.m != 0 && s < 0);
      const int32_t mi = kBf16 ? (d.m >> 16) : d.m;   // bf16: drop the 16 zero bits
      x[h] = static_cast<float>(deep ? 0 : mi);
      pw[h] = __int_as_float((deep || d.m == 0 ? 127 : s + 127) << 23);
      if (deep && gk + h < o.K && gr < o.rows) {
        const int slot = take_deep_slot(o.list_count + gr, o.cap);
        if (slot < o.cap) o.list[gr * o.cap + slot] = make_uint2(static_cast<uint32_t>(gk + h), bits[h]);
      }
    }
    uint2* dst = reinterpret_cast<uint2*>(
        o.planes + (by * nkb + int64_t(blockIdx.x)) * P * kPlaneRows * kStageK +
        r * kStageK + kq);
    write_residue_quads<0, P>(dst, x, pw);
    add_row_norm<kBf16, 16>(o, gr, x, pw);                  // a half-warp covers the row's stage
  }
}

// Fused exponent pass and residue planes, for K-contiguous rows that start on
// a vector boundary, with K <= kFusedK: one block per row, the whole row held
// in registers (four runs of four neighbouring k per thread), so the operand
// is read once.  The block takes the row's largest exponent key (one
// atomicMax per warp on a zeroed slot, read back after a barrier: no shared
// memory, so the launch for a later band can run beside a tensor-core GEMM),
// then writes the residues exactly as residue_rows_kernel does, lists the
// deep elements (a warp holding some counts them first; one holding more than
// the list's capacity writes nothing for the row), and adds the row's norm
// bound.  Once the row's norm is
// complete the block folds it into its operand's maximum; the launch's last
// block then picks the band's moduli count.  Blocks at or beyond `split`
// take o1.  Rows past `rows` (up to the plane layout's multiple of 32) get
// zero residues.
constexpr int kFusedRuns = kFusedK / (4 * kThreads);

template <int kBf16, int P, bool kGrouped>
__global__ void __launch_bounds__(kThreads) residue_fused_kernel(ResidueOperand o0, ResidueOperand o1,
                                                                  unsigned split, FusedBand fb) {
  const bool second = blockIdx.x >= split;
  const ResidueOperand& o = second ? o1 : o0;
  const int64_t r = second ? blockIdx.x - split : blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const bool live_row = r < o.rows;
  // (a strided batch's rows: groups of group_rows at group_stride)
  const int64_t row0 = kGrouped && live_row ? operand_row_offset(o, r) : 0;
  uint32_t bits[kFusedRuns][4];
  int key = 0;
  unsigned low = ~0u;                               // the smallest finite nonzero key, less one
#pragma unroll
  for (int v = 0; v < kFusedRuns; ++v) {
    const int64_t k = (int64_t(v) * kThreads + tid) * 4;
#pragma unroll
    for (int h = 0; h < 4; ++h) bits[v][h] = 0u;
    if (live_row && k < o.K) {
      if (k + 4 <= o.K) {
        if (kBf16) {
          const uint2 w = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(o.X) +
                                                               (kGrouped ? row0 : r * o.ld) + k));
          bits[v][0] = w.x << 16;
          bits[v][1] = w.x & 0xFFFF0000u;
          bits[v][2] = w.y << 16;
          bits[v][3] = w.y & 0xFFFF0000u;
        } else {
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint32_t*>(o.X) +
                                                               (kGrouped ? row0 : r * o.ld) + k));
          bits[v][0] = w.x;
          bits[v][1] = w.y;
          bits[v][2] = w.z;
          bits[v][3] = w.w;
        }
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h)
          if (k + h < o.K) bits[v][h] = load_bits<kBf16>(o.X, (kGrouped ? row0 : r * o.ld) + k + h);
      }
    }
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int kh = exp_key(bits[v][h]);           // 0 for zero and non-finite elements
      key = max(key, kh);
      low = min(low, static_cast<unsigned>(kh) - 1u);
    }
  }
  key = __reduce_max_sync(0xFFFFFFFFu, key);
  if (lane == 0 && key != 0 && live_row) atomicMax(o.keymax + r, static_cast<unsigned>(key));
  __syncthreads();                                  // every warp's maximum is in place
  const int kmax = live_row ? static_cast<int>(__ldcg(o.keymax + r)) : 0;
  if (tid == 0 && live_row) o.emax[r] = kmax != 0 ? kmax - 150 : kEmaxEmpty;
  const int em = kmax != 0 ? kmax - 150 : 0;
  // A finite element is deep when its key is below kmax - kDeepGap.  A warp
  // whose elements include one counts its deep elements first and takes
  // their list slots with one atomicAdd (nearly every warp of N(0,1) data
  // has none and skips this).  A warp that finds more deep elements than the
  // row's list holds leaves the row past the capacity, general on every tile
  // (the routing sends every tile holding it to the general tiles), so it
  // writes nothing for it: the row's planes, list and norm are never read.
  // Non-finite elements elsewhere take their slots one by one.
  const unsigned wlow = __reduce_min_sync(0xFFFFFFFFu, low);
  const bool counted = live_row && wlow != ~0u && static_cast<int>(wlow) + 1 < kmax - kDeepGap;
  int slot = 0;                                     // this thread's next list slot
  int warp_deep = 0;                                // the warp's deep elements (if counted)
  int deep_seen = 0;                                // largest list slot + 1 this thread took
  if (counted) {                                    // (the same for the whole warp)
    int mine = 0;
#pragma unroll
    for (int v = 0; v < kFusedRuns; ++v) {
      const int64_t k = (int64_t(v) * kThreads + tid) * 4;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const Decoded d = decode_f32_bits(bits[v][h]);
        const bool deep = d.nonfinite || (d.m != 0 && d.e - em + kDeepGap < 0);
        mine += deep && k + h < o.K ? 1 : 0;
      }
    }
    int incl = mine;                                // inclusive prefix over the warp
#pragma unroll
    for (int w = 1; w < 32; w *= 2) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, w);
      if (lane >= w) incl += t;
    }
    int base = 0;
    if (lane == 31 && incl > 0) base = atomicAdd(o.list_count + r, incl);
    base = __shfl_sync(0xFFFFFFFFu, base, 31);
    warp_deep = __shfl_sync(0xFFFFFFFFu, incl, 31);
    slot = base + incl - mine;
    deep_seen = base + warp_deep;                   // (the row's count once this warp's are in)
  }
  const int64_t nkb = o.Kp / kStageK;
  float sum = 0.0f;                                 // this thread's X_int^2 / 2^norm_shift
  constexpr float kHalfShift = kBf16 ? 0x1p-8f : 0x1p-26f;
  if (warp_deep <= o.cap) {                         // (the same for the whole warp)
#pragma unroll
    for (int v = 0; v < kFusedRuns; ++v) {
      const int64_t k = (int64_t(v) * kThreads + tid) * 4;
      if (k >= o.Kp) break;                         // the whole run lies past the padded K
      float x[4], pw[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const Decoded d = decode_f32_bits(bits[v][h]);
        const int sh = d.e - em + kDeepGap;
        const bool deep = d.nonfinite || (d.m != 0 && sh < 0);
        const int32_t mi = kBf16 ? (d.m >> 16) : d.m;
        x[h] = static_cast<float>(deep ? 0 : mi);
        pw[h] = __int_as_float((deep || d.m == 0 ? 127 : sh + 127) << 23);
        if (deep && k + h < o.K && live_row) {
          // a counted warp's slots in the order they were counted; else a
          // non-finite element's own
          const int at = counted ? slot++ : take_deep_slot(o.list_count + r, o.cap);
          if (at < o.cap) o.list[r * o.cap + at] = make_uint2(static_cast<uint32_t>(k + h), bits[v][h]);
          deep_seen = max(deep_seen, at + 1);
        }
        const float f = __fmul_rn(__fmul_rn(x[h], pw[h]), kHalfShift);   // exact
        sum = __fmaf_rn(f, f, sum);
      }
      uint2* dst = reinterpret_cast<uint2*>(
          o.planes + ((r / kPlaneRows) * nkb + k / kStageK) * P * kPlaneRows * kStageK +
          (r % kPlaneRows) * kStageK + (k % kStageK));
      write_residue_quads<0, P>(dst, x, pw);
    }
  }
  // the row's norm bound: 16 roundings in the thread, 5 in the warp (all to
  // nearest, positive values: relative error below 2^-19), scaled by
  // 1 + 2^-16 and converted upwards
#pragma unroll
  for (int w = 16; w >= 1; w /= 2) sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, w));
  if (lane == 0 && live_row && sum > 0.0f)
    atomicAdd(o.norm + r, __float2ull_ru(__fmul_ru(sum, 1.0f + 0x1p-16f)));
  // the row's deep count is the largest of these over its warps: one
  // atomicMax per warp that found a deep element into its 64-row block
  deep_seen = __reduce_max_sync(0xFFFFFFFFu, deep_seen);
  if (lane == 0 && deep_seen > 0 && o.dmax != nullptr)
    atomicMax(o.dmax + r / kTile, static_cast<unsigned>(deep_seen));
  __syncthreads();                                  // the row's norm and deep count are complete
  if (tid >= 32) return;
  unsigned last = 0;
  if (tid == 0) {
    if (live_row) atomicMax(o.norm_max, __ldcg(o.norm + r));
    __threadfence();
    last = atomicAdd(fb.done, 1u) == gridDim.x - 1 ? 1u : 0u;
  }
  if (__shfl_sync(0xFFFFFFFFu, last, 0) == 0u) return;
  // the launch's last block (its first warp): every row's maximum is in place
  __threadfence();
  unsigned minA = ~0u, minB = ~0u;
  if (fb.dmaxA != nullptr) {
    for (int64_t i = lane; i < fb.blocksA; i += 32) minA = min(minA, __ldcg(fb.dmaxA + i));
    for (int64_t i = lane; i < fb.blocksB; i += 32) minB = min(minB, __ldcg(fb.dmaxB + i));
    minA = __reduce_min_sync(0xFFFFFFFFu, minA);
    minB = __reduce_min_sync(0xFFFFFFFFu, minB);
  }
  if (lane != 0) return;
  const unsigned long long a = atomicAdd(const_cast<unsigned long long*>(fb.maxA), 0ull);
  const unsigned long long b = atomicAdd(const_cast<unsigned long long*>(fb.maxB), 0ull);
  int Pn = choose_moduli(a, b, fb.least, fb.most, fb.thr);
  if (fb.dmaxA != nullptr && fb.blocksA > 0 && fb.blocksB > 0 &&
      static_cast<uint64_t>(minA) + minB > static_cast<uint64_t>(fb.cap))
    Pn = 0;                                         // every tile of the band is general
  *fb.used = Pn;
  if (fb.band >= 0 && fb.band < kModuliRecord) g_moduli_record[fb.band] = Pn;
}

// ---------------------------------------------------------------- reconstruction
//
// Per output (m, n) on a residue-path tile:
//   S   = the unique integer with S = r_i (mod p_i), |S| < M/2 (M = prod p_i),
//         by the CRT sum  S' = sum_i r_i C_i,  C_i = (M/p_i) * ((M/p_i)^-1 mod p_i),
//         S = S' mod M (balanced);
//   T   = S * 2^64 plus every product involving a deep element, exact, as a
//         192-bit two's-complement integer whose bit 0 weighs 2^E with
//         E = emaxA + emaxB - 36 - 64 (+32 for bf16 planes);
//   out = RNE_f32(T * 2^E), or T placed into canonical digits.
// A deep product whose lowest bit lies below 2^E (more than 64 bits under the
// shallow grid) or that would leave the window is handled by the full
// 18-digit route instead (rare; same exact value).

typedef unsigned __int128 u128;

struct W192 {            // two's complement, word 0 least significant
  uint64_t w[3];
};

__device__ __forceinline__ void w192_add_shifted(W192& t, int64_t prod, int shift) {
  // t += prod * 2^shift, 0 <= shift <= 140, |prod| < 2^48 (mod 2^192)
  const int q = shift >> 6, r = shift & 63;
  const __int128 x = static_cast<__int128>(prod) << r;          // |x| < 2^111
  const uint64_t x0 = static_cast<uint64_t>(x);
  const uint64_t x1 = static_cast<uint64_t>(static_cast<u128>(x) >> 64);
  const uint64_t x2 = x < 0 ? ~uint64_t(0) : uint64_t(0);
  const uint64_t a0 = q == 0 ? x0 : 0;
  const uint64_t a1 = q == 0 ? x1 : (q == 1 ? x0 : 0);
  const uint64_t a2 = q == 0 ? x2 : (q == 1 ? x1 : x0);
  const u128 lo = (static_cast<u128>(t.w[1]) << 64 | t.w[0]) + (static_cast<u128>(a1) << 64 | a0);
  const uint64_t carry = lo < (static_cast<u128>(a1) << 64 | a0) ? 1u : 0u;
  t.w[0] = static_cast<uint64_t>(lo);
  t.w[1] = static_cast<uint64_t>(lo >> 64);
  t.w[2] = t.w[2] + a2 + carry;
}

// RNE_f32(t * 2^E): the binary32 rule from its definition.
__device__ __forceinline__ uint32_t round_w192(W192 t, int E) {
  const bool neg = static_cast<int64_t>(t.w[2]) < 0;
  if (neg) {
    const u128 lo = ~(static_cast<u128>(t.w[1]) << 64 | t.w[0]);
    const u128 lo1 = lo + 1;
    t.w[0] = static_cast<uint64_t>(lo1);
    t.w[1] = static_cast<uint64_t>(lo1 >> 64);
    t.w[2] = ~t.w[2] + (lo1 == 0 ? 1u : 0u);
  }
  const uint32_t sign = neg ? 0x80000000u : 0u;
  int b;
  if (t.w[2]) b = 128 + 63 - __clzll(static_cast<long long>(t.w[2]));
  else if (t.w[1]) b = 64 + 63 - __clzll(static_cast<long long>(t.w[1]));
  else if (t.w[0]) b = 63 - __clzll(static_cast<long long>(t.w[0]));
  else return 0u;                                        // exact zero -> +0
  const int lead = E + b;                                // exponent of the leading bit
  if (lead >= 128) return sign | 0x7F800000u;
  int qexp = max(lead - 23, -149);                       // exponent of one ulp
  const int s = qexp - E;                                // its bit index in t
  uint64_t q;
  if (s <= 0) {
    q = t.w[0] << (-s);                                  // exact: fewer than 24 bits
  } else {
    const int p = s - 1;                                 // index of the rounding bit
    // p >= 192: all of |t| lies below the rounding bit, below half the least
    // subnormal, so it rounds to zero (the window below is then all zero)
    const int wi = p >> 6, r = p & 63;
    const uint64_t lo = wi == 0 ? t.w[0] : (wi == 1 ? t.w[1] : (wi == 2 ? t.w[2] : 0u));
    const uint64_t hi = wi == 0 ? t.w[1] : (wi == 1 ? t.w[2] : 0u);
    const uint64_t win = r ? ((lo >> r) | (hi << (64 - r))) : lo;
    const uint64_t below_mask = r ? ((uint64_t(1) << r) - 1) : 0u;
    const bool sticky = (lo & below_mask) != 0 || (wi >= 1 && t.w[0] != 0) ||
                        (wi >= 2 && t.w[1] != 0);
    const uint64_t half = win & 1u;
    q = (win >> 1) & 0xFFFFFFu;
    if (half && (sticky || (q & 1u))) ++q;
    if (q == (uint64_t(1) << 24)) {
      q >>= 1;
      ++qexp;
    }
  }
  if (qexp > 104) return sign | 0x7F800000u;
  const uint32_t bits = q >= (uint64_t(1) << 23)
                            ? (static_cast<uint32_t>(qexp + 150) << 23) |
                                  static_cast<uint32_t>(q - (uint64_t(1) << 23))
                            : static_cast<uint32_t>(q);
  return sign | bits;
}

// d += t * 2^off (units of 2^-298); t * 2^off is a multiple of 2^-298.
__device__ __forceinline__ void add_w192_to_digits(int64_t (&d)[kDigits], W192 t, int off) {
  if (off < 0) {                                         // low bits are zero: shift exactly
    int rem = -off;                                      // shifted in steps of <= 63
    while (rem > 0) {
      const int st = rem > 63 ? 63 : rem;
      t.w[0] = (t.w[0] >> st) | (t.w[1] << (64 - st));
      t.w[1] = (t.w[1] >> st) | (t.w[2] << (64 - st));
      t.w[2] = static_cast<uint64_t>(static_cast<int64_t>(t.w[2]) >> st);
      rem -= st;
    }
    off = 0;
  }
  const int j = off >> 5, sh = off & 31;
  uint32_t x[7];
  const uint32_t sx = static_cast<int64_t>(t.w[2]) < 0 ? 0xFFFFFFFFu : 0u;
  const uint32_t wd[7] = {static_cast<uint32_t>(t.w[0]), static_cast<uint32_t>(t.w[0] >> 32),
                          static_cast<uint32_t>(t.w[1]), static_cast<uint32_t>(t.w[1] >> 32),
                          static_cast<uint32_t>(t.w[2]), static_cast<uint32_t>(t.w[2] >> 32), sx};
  x[0] = wd[0] << sh;
#pragma unroll
  for (int i = 1; i < 7; ++i) x[i] = __funnelshift_l(wd[i - 1], wd[i], sh);
  int64_t y[7];
#pragma unroll
  for (int i = 0; i < 6; ++i) y[i] = static_cast<int64_t>(x[i]);
  y[6] = static_cast<int64_t>(static_cast<int32_t>(x[6]));
#pragma unroll
  for (int pl = 0; pl < kDigits; ++pl) {
    int64_t add = 0;
#pragma unroll
    for (int i = 0; i < 7; ++i) add += (pl == j + i) ? y[i] : 0;
    // pieces above digit 17 carry only the sign extension of a value that
    // fits in 576 bits: fold them into digit 17 (mod 2^64, where a piece two
    // digits up contributes 0)
    if (pl == kDigits - 1) {
#pragma unroll
      for (int i = 0; i < 7; ++i) {
        const int over = j + i - (kDigits - 1);
        if (over == 1) add += static_cast<int64_t>(static_cast<uint64_t>(y[i]) << 32);
      }
    }
    d[pl] += add;
  }
}

__device__ __forceinline__ void add_product(int64_t (&d)[kDigits], int32_t ma, int ea, int32_t mb,
                                            int eb) {
  const int64_t prod = static_cast<int64_t>(ma) * static_cast<int64_t>(mb);
  if (prod == 0) return;
  const int off = ea + eb + kLsbBias;                    // in [0, 506]
  const uint32_t p0 = static_cast<uint32_t>(prod);
  const uint32_t p1 = static_cast<uint32_t>(static_cast<uint64_t>(prod) >> 32);
  const uint32_t sx = static_cast<uint32_t>(static_cast<int32_t>(p1) >> 31);
  const int64_t lo = static_cast<int64_t>(__funnelshift_l(0u, p0, off));
  const int64_t hi = static_cast<int64_t>(
      (static_cast<uint64_t>(__funnelshift_l(p1, sx, off)) << 32) | __funnelshift_l(p0, p1, off));
  const int j = off >> 5;
#pragma unroll
  for (int pl = 0; pl < kDigits; ++pl) d[pl] += pl == j ? lo : pl == j + 1 ? hi : 0;
}

// Bits [pos, pos+32) of the 192-bit two's-complement t (zero below bit 0,
// sign bits above bit 191).
__device__ __forceinline__ uint32_t w192_bits32(const W192& t, int pos) {
  const uint64_t sx = static_cast<int64_t>(t.w[2]) < 0 ? ~uint64_t(0) : uint64_t(0);
  if (pos <= -32) return 0u;
  if (pos < 0) return static_cast<uint32_t>(t.w[0] << (-pos));
  if (pos >= 192) return static_cast<uint32_t>(sx);
  const int w = pos >> 6, r = pos & 63;
  const uint64_t lo = w == 0 ? t.w[0] : (w == 1 ? t.w[1] : t.w[2]);
  const uint64_t hi = w == 0 ? t.w[1] : (w == 1 ? t.w[2] : sx);
  return static_cast<uint32_t>(r ? ((lo >> r) | (hi << (64 - r))) : lo);
}

// The canonical digits of t * 2^E (a multiple of 2^-298 whose magnitude is
// below 2^(575-298)) written as one output's 20 planes.
__device__ __forceinline__ void write_canonical_digits(int64_t* out, int64_t MN, W192 t, int E,
                                                       int64_t K, int64_t nf) {
  int off = E + kLsbBias;                       // bit offset of t's bit 0 in the digits
  while (off < 0) {                             // the low bits are zero: shift exactly
    const int st = -off > 63 ? 63 : -off;
    t.w[0] = (t.w[0] >> st) | (t.w[1] << (64 - st));
    t.w[1] = (t.w[1] >> st) | (t.w[2] << (64 - st));
    t.w[2] = static_cast<uint64_t>(static_cast<int64_t>(t.w[2]) >> st);
    off += st;
  }
#pragma unroll
  for (int j = 0; j < kDigits - 1; ++j)
    out[j * MN] = static_cast<int64_t>(w192_bits32(t, 32 * j - off));
  // digit 17: the signed value of bits 544 and up (fits in 32 bits)
  const int pos = 32 * (kDigits - 1) - off;
  out[(kDigits - 1) * MN] = static_cast<int64_t>(static_cast<int32_t>(w192_bits32(t, pos)));
  out[kDigits * MN] = K;
  out[(kDigits + 1) * MN] = nf;
}

// The canonical digits of S * 2^E for a signed 128-bit S = (hi:lo) (a
// multiple of 2^-298 below 2^277 in magnitude), as a window.  Digit j holds
// bits [32j - off, 32j - off + 32) of S, off = E + 298: the five words of S
// shifted by off mod 32 land on digits j0 = off/32 .. j0 + 4 (x[0..4]),
// digits below are 0 and digits above repeat the sign word sx (digits 0-16
// are unsigned words, digit 17 the signed top).
struct DigitWindow {
  int j0;
  uint32_t x[5];
  uint32_t sx;
};

__device__ __forceinline__ DigitWindow digit_window(uint64_t lo, uint64_t hi, int E) {
  int off = E + kLsbBias;
  if (off < 0) {                                // the low -off (< 64) bits are zero
    const int r = -off;
    lo = (lo >> r) | (hi << (64 - r));
    hi = static_cast<uint64_t>(static_cast<int64_t>(hi) >> r);
    off = 0;
  }
  DigitWindow d;
  d.j0 = off >> 5;
  const int sh = off & 31;
  const uint32_t w0 = static_cast<uint32_t>(lo), w1 = static_cast<uint32_t>(lo >> 32);
  const uint32_t w2 = static_cast<uint32_t>(hi), w3 = static_cast<uint32_t>(hi >> 32);
  d.sx = static_cast<uint32_t>(static_cast<int32_t>(w3) >> 31);
  d.x[0] = w0 << sh;
  d.x[1] = __funnelshift_l(w0, w1, sh);
  d.x[2] = __funnelshift_l(w1, w2, sh);
  d.x[3] = __funnelshift_l(w2, w3, sh);
  d.x[4] = __funnelshift_l(w3, d.sx, sh);
  return d;
}

// int64 value of digit plane j holding the 32-bit word w
__device__ __forceinline__ int64_t digit_of(uint32_t w, int j) {
  return j < kDigits - 1 ? static_cast<int64_t>(w) : static_cast<int64_t>(static_cast<int32_t>(w));
}

// Digit plane j's 32-bit word for a window starting at digit J0 (compile time).
template <int J0, int j>
__device__ __forceinline__ uint32_t window_word(const DigitWindow& d) {
  if constexpr (j < J0) return 0u;
  else if constexpr (j < J0 + 5) return d.x[j - J0];
  else return d.sx;
}

// One output's 20 planes; the window's start J0 is a compile-time constant, so
// every plane is one store of a known word.
// Digit planes are written once and read only by a later call: streaming
// stores, so that they do not evict what a running tensor-core GEMM shares
// through L2.
__device__ __forceinline__ void put_digit(int64_t* p, int64_t v) {
  __stcs(reinterpret_cast<long long*>(p), static_cast<long long>(v));
}

template <int J0, int j>
__device__ __forceinline__ void write_window_planes(int64_t* out, int64_t MN, const DigitWindow& d) {
  if constexpr (j < kDigits) {
    put_digit(out + j * MN, digit_of(window_word<J0, j>(d), j));
    write_window_planes<J0, j + 1>(out, MN, d);
  }
}

template <int J0>
__device__ __forceinline__ void write_window_at(int64_t* out, int64_t MN, const DigitWindow& d, int64_t K,
                                                int64_t nf) {
  write_window_planes<J0, 0>(out, MN, d);
  put_digit(out + kDigits * MN, K);
  put_digit(out + (kDigits + 1) * MN, nf);
}

// The same for any start, in the general form (words selected at run time).
__device__ __forceinline__ void write_window_any(int64_t* out, int64_t MN, const DigitWindow& d,
                                                 int64_t K, int64_t nf) {
#pragma unroll
  for (int j = 0; j < kDigits; ++j) {
    const int k = j - d.j0;
    const uint32_t w = k < 0 ? 0u
                     : k == 0 ? d.x[0] : k == 1 ? d.x[1] : k == 2 ? d.x[2] : k == 3 ? d.x[3]
                     : k == 4 ? d.x[4] : d.sx;
    put_digit(out + j * MN, digit_of(w, j));
  }
  put_digit(out + kDigits * MN, K);
  put_digit(out + (kDigits + 1) * MN, nf);
}

// Dispatch on the window's start.  For finite operands it is at most 14
// (E <= 2 * 104 - 38, so off = E + 298 < 480); larger starts take the
// general form.
__device__ __forceinline__ void write_window(int64_t* out, int64_t MN, const DigitWindow& d, int64_t K,
                                             int64_t nf) {
  switch (d.j0) {
#define DET_WINDOW_CASE(J) \
  case J: write_window_at<J>(out, MN, d, K, nf); break;
    DET_WINDOW_CASE(0) DET_WINDOW_CASE(1) DET_WINDOW_CASE(2) DET_WINDOW_CASE(3)
    DET_WINDOW_CASE(4) DET_WINDOW_CASE(5) DET_WINDOW_CASE(6) DET_WINDOW_CASE(7)
    DET_WINDOW_CASE(8) DET_WINDOW_CASE(9) DET_WINDOW_CASE(10) DET_WINDOW_CASE(11)
    DET_WINDOW_CASE(12) DET_WINDOW_CASE(13) DET_WINDOW_CASE(14)
#undef DET_WINDOW_CASE
    default: write_window_any(out, MN, d, K, nf);
  }
}

// Cold path of one output: the digit route.  Used for det_gemm_partial (the
// digits are the output) and when a deep product falls outside the 192-bit
// window; rebuilds the exact value as 18 int64 digits and writes it.
template <int kBf16>
__device__ __noinline__ void output_via_digits(const GemmArgs& g, const ReconArgs& ra, int64_t m,
                                               int64_t n, int64_t sb, W192 t, int E, bool wide,
                                               __int128 S, int emA, int64_t nf) {
  const int64_t MN = g.M * g.N;
  int64_t d[kDigits];
#pragma unroll
  for (int pl = 0; pl < kDigits; ++pl) d[pl] = 0;
  if (!wide) {
    add_w192_to_digits(d, t, E + kLsbBias);
  } else {
    W192 s0;
    s0.w[0] = 0;
    s0.w[1] = static_cast<uint64_t>(S);
    s0.w[2] = static_cast<uint64_t>(S >> 64);
    add_w192_to_digits(d, s0, E + kLsbBias);
    const int na = min(ra.countA[m], ra.cap);
    const int nb = min(ra.countB[sb], ra.cap);
    for (int q = 0; q < na; ++q) {
      const uint2 ent = ra.listA[m * ra.cap + q];
      const int64_t k = ent.x;
      const Decoded a = decode_f32_bits(ent.y);
      const Decoded b = decode_f32_bits(load_bits<kBf16>(g.B, b_offset(g, sb, k)));
      if (!a.nonfinite && !b.nonfinite) add_product(d, a.m, a.e, b.m, b.e);
    }
    for (int q = 0; q < nb; ++q) {
      const uint2 ent = ra.listB[sb * ra.cap + q];
      const int64_t k = ent.x;
      const Decoded b = decode_f32_bits(ent.y);
      const Decoded a = decode_f32_bits(load_bits<kBf16>(g.A, a_offset(g, m, k)));
      if (a.nonfinite || (a.m != 0 && a.e - emA + kDeepGap < 0)) continue;
      if (!b.nonfinite) add_product(d, a.m, a.e, b.m, b.e);
    }
  }
  uint32_t w[kDigits - 1];
  int64_t top;
  normalise_digits(d, w, top);
  if (g.P) {
    int64_t* out = g.P + m * g.N + n;
#pragma unroll
    for (int pl = 0; pl < kDigits - 1; ++pl) out[pl * MN] = static_cast<int64_t>(w[pl]);
    out[(kDigits - 1) * MN] = top;
    out[kDigits * MN] = g.K;
    out[(kDigits + 1) * MN] = nf;
  } else {
    reinterpret_cast<uint32_t*>(g.C)[c_row_offset(g, m) + n] = nf ? kNanBits : round_to_f32_bits(w, top);
  }
}

// ---------------------------------------------------------------- CRT
//
// The residue GEMM stores balanced residues r_i (|r_i| <= (p_i - 1)/2) as
// two's-complement bytes.  The reconstruction rebuilds S as one sum of
// products, crt_s128 (det_crt.cuh): about 60 integer multiply-adds per
// output, with compile-time constants for each count of moduli.

// Byte j of a word of four residue bytes, sign-extended: one byte permute
// whose selector copies byte j and replicates its sign bit into the three
// bytes above (a selector nibble with its top bit set; __byte_perm keeps only
// the low three bits of each nibble, so the instruction is written out).
__device__ __forceinline__ int32_t residue_of_word(uint32_t w, int j) {
  const uint32_t sj = 8u | static_cast<uint32_t>(j);
  const uint32_t sel = (sj << 12) | (sj << 8) | (sj << 4) | static_cast<uint32_t>(j);
  uint32_t d;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(w), "r"(sel));
  return static_cast<int32_t>(d);
}

// RNE_f32(S * 2^E) for a signed 128-bit S = (hi:lo): the binary32 rule,
// bit by bit.  Used where the result may be subnormal.
__device__ __noinline__ uint32_t round_s128_exact(uint64_t lo, uint64_t hi, int E) {
  const bool neg = static_cast<int64_t>(hi) < 0;
  if (neg) {
    lo = ~lo + 1;
    hi = ~hi + (lo == 0 ? 1u : 0u);
  }
  const uint32_t sign = neg ? 0x80000000u : 0u;
  int b;
  if (hi) b = 64 + 63 - __clzll(static_cast<long long>(hi));
  else if (lo) b = 63 - __clzll(static_cast<long long>(lo));
  else return 0u;                                        // exact zero -> +0
  const int lead = E + b;
  if (lead >= 128) return sign | 0x7F800000u;
  int qexp = max(lead - 23, -149);
  const int s = qexp - E;                                // bit index of one ulp
  uint64_t q;
  if (s <= 0) {
    q = lo << (-s);                                      // exact (fewer than 24 bits)
  } else {
    const int p = s - 1;                                 // rounding bit
    uint64_t win;
    bool sticky;
    if (p < 64) {
      win = p ? ((lo >> p) | (hi << (64 - p))) : lo;
      sticky = p ? (lo & ((uint64_t(1) << p) - 1)) != 0 : false;
    } else if (p < 128) {
      const int p2 = p - 64;
      win = hi >> p2;
      sticky = lo != 0 || (p2 ? (hi & ((uint64_t(1) << p2) - 1)) != 0 : false);
    } else {                                             // all of |S| lies below the rounding
      win = 0;                                           // bit: below half the least
      sticky = true;                                     // subnormal, so it rounds to zero
    }
    const uint64_t half = win & 1u;
    q = (win >> 1) & 0xFFFFFFu;
    if (half && (sticky || (q & 1u))) ++q;
    if (q == (uint64_t(1) << 24)) {
      q >>= 1;
      ++qexp;
    }
  }
  if (qexp > 104) return sign | 0x7F800000u;
  const uint32_t bits = q >= (uint64_t(1) << 23)
                            ? (static_cast<uint32_t>(qexp + 150) << 23) |
                                  static_cast<uint32_t>(q - (uint64_t(1) << 23))
                            : static_cast<uint32_t>(q);
  return sign | bits;
}

// RNE_f32(S * 2^E), fast form.  The leading 64 bits of |S|, with every bit
// below them ORed into bit 0 (a sticky bit well below the rounding position),
// round to binary32 with the same round-to-nearest-even decision as |S|
// itself; the exact power-of-two scaling is then an exponent add.  Results
// that would be subnormal or zero go to the bit-by-bit routine.
__device__ __forceinline__ uint32_t round_s128(uint64_t lo, uint64_t hi, int E) {
  const bool neg = static_cast<int64_t>(hi) < 0;
  uint64_t alo = lo, ahi = hi;
  if (neg) {
    alo = ~lo + 1;
    ahi = ~hi + (alo == 0 ? 1u : 0u);
  }
  if ((alo | ahi) == 0) return 0u;                       // exact zero -> +0
  const int lz = ahi ? __clzll(static_cast<long long>(ahi))
                     : 64 + __clzll(static_cast<long long>(alo));
  uint64_t top;
  if (lz == 0) {
    top = ahi | (alo != 0 ? 1u : 0u);
  } else if (lz < 64) {
    top = (ahi << lz) | (alo >> (64 - lz)) | ((alo << lz) != 0 ? 1u : 0u);
  } else {
    top = alo << (lz - 64);
  }
  const uint32_t f = f32_bits_of_top(top);                      // |S| * 2^(lz-64), rounded
  const int shift = E + 64 - lz;
  const int ef = static_cast<int>(f >> 23) + shift;             // biased exponent of the result
  if (ef >= 1 && ef <= 254) return (neg ? 0x80000000u : 0u) | (f + (static_cast<uint32_t>(shift) << 23));
  if (ef >= 255) return (neg ? 0x80000000u : 0u) | 0x7F800000u;
  return round_s128_exact(lo, hi, E);
}

// Deep products of output (m, n) added into t (bit 0 weighs 2^E); returns
// false if one of them does not fit the window (the caller then takes the
// digit route).  nf counts products with a non-finite operand.
template <int kBf16>
__device__ __noinline__ bool add_deep_products(const GemmArgs& g, const ReconArgs& ra, int64_t m,
                                               int64_t sb, int emA, int E, W192& t, int64_t& nf) {
  // sb: B's row of the output's column (its stacked row in a strided batch)
  bool fits = true;
  const int na = min(ra.countA[m], ra.cap);
  const int nb = min(ra.countB[sb], ra.cap);
  for (int q = 0; q < na; ++q) {                 // row m of A's deep elements x column n of B
    const uint2 ent = ra.listA[m * ra.cap + q];
    const int64_t k = ent.x;
    const Decoded a = decode_f32_bits(ent.y);
    const Decoded b = decode_f32_bits(load_bits<kBf16>(g.B, b_offset(g, sb, k)));
    if (a.nonfinite || b.nonfinite) {
      ++nf;
    } else if (a.m != 0 && b.m != 0) {
      const int sh = a.e + b.e - E;
      if (sh < 0 || sh > 140) fits = false;
      else w192_add_shifted(t, static_cast<int64_t>(a.m) * b.m, sh);
    }
  }
  for (int q = 0; q < nb; ++q) {                 // column n of B's deep elements x shallow row m
    const uint2 ent = ra.listB[sb * ra.cap + q];
    const int64_t k = ent.x;
    const Decoded b = decode_f32_bits(ent.y);
    const Decoded a = decode_f32_bits(load_bits<kBf16>(g.A, a_offset(g, m, k)));
    if (a.nonfinite || (a.m != 0 && a.e - emA + kDeepGap < 0)) continue;   // row m's list had it
    if (b.nonfinite) {
      ++nf;
    } else if (a.m != 0 && b.m != 0) {
      const int sh = a.e + b.e - E;
      if (sh < 0 || sh > 140) fits = false;
      else w192_add_shifted(t, static_cast<int64_t>(a.m) * b.m, sh);
    }
  }
  return fits;
}

// Calls f with the moduli count `used` as a compile-time constant, for
// counts from the least compiled one up to P (a count outside that range
// takes the nearer end; the host never passes one).
template <int kBf16, int P, typename F>
__device__ __forceinline__ void with_used_planes(int used, F&& f) {
  if constexpr (P > planes_least(kBf16)) {
    if (used < P) {
      with_used_planes<kBf16, P - 1>(used, f);
      return;
    }
  }
  f(std::integral_constant<int, P>{});
}

constexpr int kReconCols = 4;                       // outputs per thread (one row)

// Fast path: det_gemm outputs whose row of A and column of B hold no deep
// element -- CRT, then one rounding.  Nothing else, to keep registers low.
template <int kBf16, int P, bool kGrouped>
__device__ __forceinline__ void reconstruct_fast_body(const GemmArgs& g, const ReconArgs& ra) {
  const int64_t MN = g.M * g.N;
  const int64_t tiles_n = (g.N + kTile - 1) / kTile;
  const bool failed = ra.error != nullptr && *ra.error != 0;    // the tensor-core kernel gave up
  const int64_t n0 = (int64_t(blockIdx.x) * kThreads + threadIdx.x) * kReconCols;
  if (n0 >= g.N) return;
  const int ncols = g.N - n0 < kReconCols ? static_cast<int>(g.N - n0) : kReconCols;
  const bool vec_ok = ((MN & 3) == 0) && ((g.N & 3) == 0) &&
                      (reinterpret_cast<uintptr_t>(ra.res) & 3u) == 0;
  // the thread's columns' deep flags and exponents: once, or (a strided
  // batch) once per entry its rows reach
  uint32_t live = 0;                     // bit j: column n0 + j is reconstructed here
  int colE[kReconCols];
  auto columns_of = [&](int64_t e) {
    live = 0;
#pragma unroll
    for (int j = 0; j < kReconCols; ++j) {
      colE[j] = 0;
      if (j < ncols) {
        const int64_t n = e * g.N + n0 + j;                       // B's stacked row
        if (ra.countB[n] == 0) live |= 1u << j;                   // else: deep kernel
        int emB = ra.emaxB[n];
        emB = emB == kEmaxEmpty ? 0 : emB;
        colE[j] = emB - 2 * kDeepGap + (kBf16 ? 32 : 0);
      }
    }
  };
  int64_t entry = 0;
  if constexpr (kGrouped) entry = entry_div(ra.m_begin + int64_t(blockIdx.y), g.Me);
  columns_of(entry);
  if (!kGrouped && live == 0) return;
  // all four outputs of a row in one 16-byte store where the layout allows
  static_assert(kReconCols == 4, "one uint4 of outputs per row");
  const bool store4_ok = (g.ldc & 3) == 0 && (reinterpret_cast<uintptr_t>(g.C) & 15u) == 0 &&
                         (!kGrouped || (g.strideC & 3) == 0);
  const bool store4 = store4_ok && live == (1u << kReconCols) - 1;   // (fixed columns)
  const bool vec = vec_ok && ncols == kReconCols;
  auto load_row = [&](int64_t m, uint32_t (&packed)[kNumModuli]) {
    const int64_t base = m * g.N + n0;
#pragma unroll
    for (int i = 0; i < kNumModuli; ++i) {
      packed[i] = 0;
      if (i < P) {
        const int8_t* plane = ra.res + i * MN + base;
        if (vec) {
          packed[i] = __ldcs(reinterpret_cast<const unsigned int*>(plane));   // read once
        } else {
#pragma unroll
          for (int j = 0; j < kReconCols; ++j)
            if (j < ncols) packed[i] |= static_cast<uint32_t>(static_cast<uint8_t>(plane[j])) << (8 * j);
        }
      }
    }
  };
  auto finish_row = [&](int64_t m, const uint32_t (&packed)[kNumModuli]) {
    if constexpr (kGrouped) {
      const int64_t e = entry_div(m, g.Me);
      if (e != entry) {
        entry = e;
        columns_of(e);
      }
      if (live == 0) return;
    }
    if (ra.route[(m / kTile) * tiles_n + n0 / kTile]) return;     // general kernel's outputs
    if (ra.countA[m] != 0) return;                                // deep row: deep kernel
    int emA = ra.emaxA[m];
    emA = emA == kEmaxEmpty ? 0 : emA;
    uint32_t out[kReconCols];
#pragma unroll
    for (int j = 0; j < kReconCols; ++j) {
      out[j] = kNanBits;
      if (((live >> j) & 1u) == 0u) continue;
      int32_t r[kNumModuli];
#pragma unroll
      for (int i = 0; i < kNumModuli; ++i) r[i] = residue_of_word(packed[i], j);
      uint64_t slo, shi;
      crt_s128<P>(r, slo, shi);
      if (!failed) out[j] = round_s128(slo, shi, emA + colE[j]);
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>(g.C) + (kGrouped ? c_row_offset(g, m) : m * g.ldc) + n0;
    if (kGrouped ? store4_ok && live == (1u << kReconCols) - 1 : store4) {
      __stcs(reinterpret_cast<uint4*>(dst), make_uint4(out[0], out[1], out[2], out[3]));
    } else {
#pragma unroll
      for (int j = 0; j < kReconCols; ++j)
        if ((live >> j) & 1u) dst[j] = out[j];
    }
  };
  // two rows per step: both rows' residue loads are in flight before either
  // row's arithmetic
  const int64_t step = gridDim.y;
  for (int64_t m = ra.m_begin + blockIdx.y; m < ra.m_end; m += 2 * step) {
    const bool two = m + step < ra.m_end;
    uint32_t p0[kNumModuli], p1[kNumModuli];
    load_row(m, p0);
    if (two) load_row(m + step, p1);
    finish_row(m, p0);
    if (two) finish_row(m + step, p1);
  }
}

// The launch is compiled for the planes' count P and runs the body for the
// band's count (ReconArgs::used).
template <int kBf16, int P, bool kGrouped>
__global__ void __launch_bounds__(kThreads, 4) reconstruct_fast_kernel(GemmArgs g, ReconArgs ra) {
  if (ra.used != nullptr && *ra.used == 0) return;   // every tile of the band is general
  with_used_planes<kBf16, P>(ra.used ? *ra.used : P, [&](auto Q) {
    reconstruct_fast_body<kBf16, decltype(Q)::value, kGrouped>(g, ra);
  });
}

// Outputs with deep entries: every output of a deep row, then every output of
// a deep column outside the deep rows.  Dense work list, so the warps stay
// full.  It shares nothing with the fast kernels but the residues (read
// only), so it runs beside them.
template <int kBf16, int P>
__device__ __forceinline__ void reconstruct_deep_body(const GemmArgs& g, const ReconArgs& ra,
                                                      const int* rows, const int* cols,
                                                      const int* nrc, int parts) {
  const int64_t MN = g.M * g.N;
  const int64_t tiles_n = (g.N + kTile - 1) / kTile;
  const bool failed = ra.error != nullptr && *ra.error != 0;
  const int64_t n_rows = (parts & kDeepRows) ? nrc[0] : 0;
  const int64_t n_cols = (parts & kDeepCols) ? nrc[1] : 0;
  const int64_t band = ra.m_end - ra.m_begin;
  // the deep-column part walks, per listed column, the band's rows; in a
  // strided batch the listed columns are B's stacked rows e * N + n, and
  // only entry e's rows (those in the band) take them
  const bool grouped = g.batch > 1;
  const int64_t col_rows = grouped ? g.Me : band;
  const int64_t part1 = n_rows * g.N, total = part1 + col_rows * n_cols;
  for (int64_t idx = int64_t(blockIdx.x) * kThreads + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * kThreads) {
    int64_t m, n, sb;
    if (idx < part1) {
      m = rows[idx / g.N];
      if (m < ra.m_begin || m >= ra.m_end) continue;              // another band's row
      n = idx - (idx / g.N) * g.N;
      sb = brow_of(g, m, n);
    } else {
      const int64_t j = idx - part1;
      const int64_t mb = j / n_cols;
      sb = cols[j - mb * n_cols];
      if (grouped) {
        const int64_t e = entry_div(sb, g.N);
        n = sb - e * g.N;
        m = e * g.Me + mb;
        if (m < ra.m_begin || m >= ra.m_end) continue;            // another band's entry
      } else {
        m = ra.m_begin + mb;
        n = sb;
      }
      if (ra.countA[m] != 0) continue;                          // done with its deep row
    }
    if (ra.route[(m / kTile) * tiles_n + n / kTile]) continue;  // general kernel's output
    int emA = ra.emaxA[m], emB = ra.emaxB[sb];
    emA = emA == kEmaxEmpty ? 0 : emA;
    emB = emB == kEmaxEmpty ? 0 : emB;
    int32_t r[kNumModuli];
#pragma unroll
    for (int i = 0; i < kNumModuli; ++i) r[i] = i < P ? static_cast<int32_t>(ra.res[i * MN + m * g.N + n]) : 0;
    uint64_t slo, shi;
    crt_s128<P>(r, slo, shi);
    const int E = emA + emB - 2 * kDeepGap + (kBf16 ? 32 : 0) - 64;
    W192 t;
    t.w[0] = 0;
    t.w[1] = slo;
    t.w[2] = shi;
    int64_t nf = 0;
    const bool fits = add_deep_products<kBf16>(g, ra, m, sb, emA, E, t, nf);
    if (failed) nf = 1;
    if (fits && g.P != nullptr) {
      write_canonical_digits(g.P + m * g.N + n, MN, t, E, g.K, nf);
    } else if (fits) {
      reinterpret_cast<uint32_t*>(g.C)[c_row_offset(g, m) + n] = nf ? kNanBits : round_w192(t, E);
    } else {
      const __int128 S = static_cast<__int128>((static_cast<unsigned __int128>(shi) << 64) | slo);
      output_via_digits<kBf16>(g, ra, m, n, sb, t, E, true, S, emA, nf);
    }
  }
}

template <int kBf16, int P>
__global__ void __launch_bounds__(kThreads, 1) reconstruct_deep_kernel(
    GemmArgs g, ReconArgs ra, const int* rows, const int* cols, const int* nrc, int parts) {
  if (ra.used != nullptr && *ra.used == 0) return;   // every tile of the band is general
  with_used_planes<kBf16, P>(ra.used ? *ra.used : P, [&](auto Q) {
    reconstruct_deep_body<kBf16, decltype(Q)::value>(g, ra, rows, cols, nrc, parts);
  });
}

// det_gemm_partial outputs whose row of A and column of B hold no deep
// element: CRT, then the digits.  One output per thread, so that each of the
// 20 plane stores of a warp is one contiguous 256-byte write; the digit
// window's start selects straight-line code with one store per plane.
template <int kBf16, int P>
__device__ __forceinline__ void partial_fast_body(const GemmArgs& g, const ReconArgs& ra) {
  const int64_t MN = g.M * g.N;
  const int64_t tiles_n = (g.N + kTile - 1) / kTile;
  const int64_t nf = ra.error != nullptr && *ra.error != 0 ? 1 : 0;   // tensor-core kernel gave up
  const int64_t n = int64_t(blockIdx.x) * kThreads + threadIdx.x;
  if (n >= g.N) return;
  if (ra.countB[n] != 0) return;                              // deep column: deep kernel
  int emB = ra.emaxB[n];
  emB = emB == kEmaxEmpty ? 0 : emB;
  const int colE = emB - 2 * kDeepGap + (kBf16 ? 32 : 0);
  // two rows per step: both rows' residue loads are in flight before either
  // row's arithmetic and stores
  const int64_t step = gridDim.y;
  for (int64_t m = ra.m_begin + blockIdx.y; m < ra.m_end; m += 2 * step) {
    const bool two = m + step < ra.m_end;
    int32_t r[2][kNumModuli];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t idx = (m + h * step) * g.N + n;
#pragma unroll
      for (int i = 0; i < kNumModuli; ++i)
        r[h][i] = i < P && (h == 0 || two) ? static_cast<int32_t>(ra.res[i * MN + idx]) : 0;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t mh = m + h * step;
      if (h == 1 && !two) break;
      if (ra.route[(mh / kTile) * tiles_n + n / kTile]) continue;  // general kernel's outputs
      if (ra.countA[mh] != 0) continue;                            // deep row: deep kernel
      int emA = ra.emaxA[mh];
      emA = emA == kEmaxEmpty ? 0 : emA;
      uint64_t slo, shi;
      crt_s128<P>(r[h], slo, shi);
      const DigitWindow d = digit_window(slo, shi, emA + colE);
      write_window(g.P + mh * g.N + n, MN, d, g.K, nf);
    }
  }
}

template <int kBf16, int P>
__global__ void __launch_bounds__(kThreads, 4) partial_fast_kernel(GemmArgs g, ReconArgs ra) {
  if (ra.used != nullptr && *ra.used == 0) return;   // every tile of the band is general
  with_used_planes<kBf16, P>(ra.used ? *ra.used : P,
                             [&](auto Q) { partial_fast_body<kBf16, decltype(Q)::value>(g, ra); });
}

// The same outputs written by bulk copies.  A block owns 128 columns of a
// contiguous chunk of the band's rows.  The rows' residues, every modulus,
// arrive by 16-byte cp.async copies into a ring of kRing row buffers,
// kRing - 1 rows ahead (one thread of the block also copies the row's deep
// count and exponent maximum); each thread rebuilds its output's 20 digit
// words into shared memory, and 20 threads send the row segment's 20 planes
// (1 KB each) to global memory as bulk copies, double-buffered so that the
// next row is rebuilt while they drain.  The SMs issue 0.16 store
// instructions per output instead of 20.
//
// A bulk copy writes the whole segment, so deep columns get placeholder
// zeros: the band's deep kernel, ordered after this one, writes them.  Deep
// rows are skipped whole (the deep kernel's), and a row segment that touches
// a general tile (the general or wide kernel's outputs) is written output by
// output instead.  Needs N a multiple of 16 and 16-byte aligned residues and
// digit planes (every copy 16-byte aligned, every size a multiple of 128
// bytes); 43 KB of shared memory, five blocks per SM.
constexpr int kRing = 3;
constexpr int kBulkCols = 128;
constexpr int kPlanesOut = kDigits + 2;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

// One output's 20 plane words into column t of a shared segment buffer.
template <int J0, int j>
__device__ __forceinline__ void window_to_smem(int64_t (*seg)[kBulkCols], int t, const DigitWindow& d) {
  if constexpr (j < kDigits) {
    seg[j][t] = digit_of(window_word<J0, j>(d), j);
    window_to_smem<J0, j + 1>(seg, t, d);
  }
}
__device__ __forceinline__ void window_to_smem_any(int64_t (*seg)[kBulkCols], int t, const DigitWindow& d) {
#pragma unroll
  for (int j = 0; j < kDigits; ++j) {
    const int k = j - d.j0;
    const uint32_t w = k < 0 ? 0u
                     : k == 0 ? d.x[0] : k == 1 ? d.x[1] : k == 2 ? d.x[2] : k == 3 ? d.x[3]
                     : k == 4 ? d.x[4] : d.sx;
    seg[j][t] = digit_of(w, j);
  }
}
__device__ __forceinline__ void window_to_smem_at(int64_t (*seg)[kBulkCols], int t, const DigitWindow& d) {
  switch (d.j0) {
#define DET_SEG_CASE(J) \
  case J: window_to_smem<J, 0>(seg, t, d); break;
    DET_SEG_CASE(0) DET_SEG_CASE(1) DET_SEG_CASE(2) DET_SEG_CASE(3) DET_SEG_CASE(4)
    DET_SEG_CASE(5) DET_SEG_CASE(6) DET_SEG_CASE(7) DET_SEG_CASE(8) DET_SEG_CASE(9)
    DET_SEG_CASE(10) DET_SEG_CASE(11) DET_SEG_CASE(12) DET_SEG_CASE(13) DET_SEG_CASE(14)
#undef DET_SEG_CASE
    default: window_to_smem_any(seg, t, d);
  }
}

struct BulkSmem {
  int64_t seg[2][kDigits][kBulkCols];         // 36 KB: two row segments of digit planes
  int64_t fixed[2][kBulkCols];                // planes 18 and 19 (K, the non-finite count):
                                              //   the same in every segment of the call
  int8_t res[kRing][kNumModuli][kBulkCols];   // 5.25 KB: residue rows
  int meta[kRing][2];                         // deep count, exponent maximum of the row
};
constexpr int kBulkBlocksPerSm = 5;           // 43.3 KB each

template <int kBf16, int P>
__device__ __forceinline__ void partial_bulk_body(const GemmArgs& g, const ReconArgs& ra, BulkSmem& sm) {
  const int64_t MN = g.M * g.N;
  const int64_t tiles_n = (g.N + kTile - 1) / kTile;
  const int64_t band = ra.m_end - ra.m_begin;
  const int64_t chunk = (band + gridDim.y - 1) / gridDim.y;
  const int64_t r0 = ra.m_begin + int64_t(blockIdx.y) * chunk;
  const int64_t r1 = r0 + chunk < ra.m_end ? r0 + chunk : ra.m_end;
  if (r0 >= r1) return;                                         // the same for the whole block
  const int64_t nf = ra.error != nullptr && *ra.error != 0 ? 1 : 0;   // tensor-core kernel gave up
  const int t = threadIdx.x;
  const int64_t n0 = int64_t(blockIdx.x) * kBulkCols;
  const int64_t n = n0 + t;
  const int ncols = g.N - n0 < kBulkCols ? static_cast<int>(g.N - n0) : kBulkCols;
  const bool in_range = t < ncols;
  const bool col_live = in_range && ra.countB[n] == 0;          // deep column: deep kernel
  int colE = 0;
  if (col_live) {
    int emB = ra.emaxB[n];
    emB = emB == kEmaxEmpty ? 0 : emB;
    colE = emB - 2 * kDeepGap + (kBf16 ? 32 : 0);
  }
  // residue copies: 8 threads per modulus row of 128 bytes; two more threads
  // copy the row's metadata
  const int cu = t >> 3, cc = (t & 7) * 16;
  const bool copier = cu < P && cc < ncols;
  const int8_t* src = ra.res + cu * MN + n0 + cc;
  sm.fixed[0][t] = g.K;
  sm.fixed[1][t] = nf;
  ptx::fence_proxy_async_smem();                // read by the bulk copies (after a barrier)
  auto issue = [&](int64_t m, int slot) {
    if (m < r1) {
      if (copier) cp_async16(&sm.res[slot][cu][cc], src + m * g.N);
      if (t == kBulkCols - 1) cp_async4(&sm.meta[slot][0], ra.countA + m);
      if (t == kBulkCols - 2) cp_async4(&sm.meta[slot][1], ra.emaxA + m);
    }
    cp_async_commit();                                          // one group per row, empty or not
  };
#pragma unroll
  for (int i = 0; i < kRing - 1; ++i) issue(r0 + i, i);
  // this thread's route byte, for the current 64-row tile and the next
  const int64_t tn = (in_range ? n : n0) / kTile;
  int64_t tile_row = r0 / kTile;
  uint8_t rt = ra.route[tile_row * tiles_n + tn];
  uint8_t rt_next = (tile_row + 1) * kTile < g.M ? ra.route[(tile_row + 1) * tiles_n + tn] : 0;
  int slot = 0, oslot = 0;
  for (int64_t m = r0; m < r1; ++m) {
    if (m / kTile != tile_row) {
      ++tile_row;
      rt = rt_next;
      rt_next = (tile_row + 1) * kTile < g.M ? ra.route[(tile_row + 1) * tiles_n + tn] : 0;
    }
    // the buffers alternate by send and every send is one bulk group per
    // issuing thread: the send before last, which used the buffer this row
    // may fill, must have read it (the last one may still be reading)
    if (t < kPlanesOut) ptx::bulk_wait_read<1>();
    cp_async_wait<kRing - 2>();                   // this thread's copies of row m have landed
    const bool general = __syncthreads_or(in_range && rt != 0) != 0;   // and everyone's
    issue(m + kRing - 1, slot == 0 ? kRing - 1 : slot - 1);   // row m - 1's slot is free
    const int cA = sm.meta[slot][0];
    const int emA = sm.meta[slot][1] == kEmaxEmpty ? 0 : sm.meta[slot][1];
    if (cA == 0) {                                              // deep rows: the deep kernel's
      DigitWindow d;
      if (col_live && (!general || !rt)) {
        int32_t r[kNumModuli];
#pragma unroll
        for (int i = 0; i < kNumModuli; ++i) r[i] = i < P ? static_cast<int32_t>(sm.res[slot][i][t]) : 0;
        uint64_t slo, shi;
        crt_s128<P>(r, slo, shi);
        d = digit_window(slo, shi, emA + colE);
      } else {
        d.j0 = 0;                                   // placeholder zeros (a deep column)
        d.x[0] = d.x[1] = d.x[2] = d.x[3] = d.x[4] = 0u;
        d.sx = 0u;
      }
      if (!general) {
        if (in_range) {
          window_to_smem_at(sm.seg[oslot], t, d);
          ptx::fence_proxy_async_smem();          // visible to the bulk copies
        }
        __syncthreads();
        if (t < kPlanesOut) {
          const int64_t* from = t < kDigits ? &sm.seg[oslot][t][0] : &sm.fixed[t - kDigits][0];
          ptx::bulk_store(g.P + t * MN + m * g.N + n0, from, static_cast<uint32_t>(ncols) * 8u);
          ptx::bulk_commit();
        }
        oslot ^= 1;
      } else if (col_live && !rt) {
        write_window(g.P + m * g.N + n, MN, d, g.K, nf);        // beside a general tile
      }
    }
    slot = slot == kRing - 1 ? 0 : slot + 1;
  }
  cp_async_wait<0>();                             // nothing left in flight at exit
  if (t < kPlanesOut) ptx::bulk_wait_all();       // the copies have read shared memory
}

template <int kBf16, int P>
__global__ void __launch_bounds__(kBulkCols, kBulkBlocksPerSm) partial_bulk_kernel(GemmArgs g, ReconArgs ra) {
  if (ra.used != nullptr && *ra.used == 0) return;   // every tile of the band is general
  __shared__ __align__(128) BulkSmem sm;
  with_used_planes<kBf16, P>(ra.used ? *ra.used : P, [&](auto Q) {
    partial_bulk_body<kBf16, decltype(Q)::value>(g, ra, sm);
  });
}

// Moduli counts with compiled kernels: f32 operands need 12 to 14 moduli
// (K from 1 to 2^19), bf16 operands 8 to 10.  A call uses the smallest
// compiled count that covers its bound (more moduli never change the result).
template <typename F>
cudaError_t with_planes(int bf16, int P, F&& launch) {
  using std::integral_constant;
  if (bf16) {
    switch (P) {
      case 8: return launch(integral_constant<int, 1>{}, integral_constant<int, 8>{});
      case 9: return launch(integral_constant<int, 1>{}, integral_constant<int, 9>{});
      case 10: return launch(integral_constant<int, 1>{}, integral_constant<int, 10>{});
      default: return cudaErrorInvalidValue;
    }
  }
  switch (P) {
    case 12: return launch(integral_constant<int, 0>{}, integral_constant<int, 12>{});
    case 13: return launch(integral_constant<int, 0>{}, integral_constant<int, 13>{});
    case 14: return launch(integral_constant<int, 0>{}, integral_constant<int, 14>{});
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int residue_planes_needed(const GemmArgs& g) {
  // |S| <= K * maxA * maxB with max = (2^bits - 1) * 2^18.  The CRT sum needs
  // prod > 2|S| (1 + 2^-7): the margin lets its fixed-point quotient round
  // to the right integer (crt_s128).
  const unsigned __int128 sig = g.bf16 ? 0xFFu : 0xFFFFFFu;
  const unsigned __int128 mx = sig << kDeepGap;
  const unsigned __int128 twice = static_cast<unsigned __int128>(g.K > 0 ? g.K : 1) * mx * mx * 2;
  const unsigned __int128 bound = twice + (twice >> 7);
  unsigned __int128 prod = 1;
  const int least = planes_least(g.bf16);
  for (int i = 0; i < kNumModuli; ++i) {
    prod *= static_cast<unsigned>(modulus(i));
    if (prod > bound) return i + 1 < least ? least : i + 1;
  }
  return -1;
}

int residue_planes_least(int bf16) { return planes_least(bf16); }

ModuliThresholds moduli_thresholds(int bf16) {
  // every step below rounds to nearest in double (relative error below
  // 2^-48 in all); the factor 1 - 2^-40 keeps each threshold under the exact
  // quotient, and the conversion to a 128-bit integer is exact
  ModuliThresholds t{};
  double prod = 1.0;
  for (int P = 1; P <= kNumModuli; ++P) {
    prod *= static_cast<double>(modulus(P - 1));
    const double q = prod * prod / ldexp(1.0, 2 * norm_shift(bf16) + 2) / (129.0 / 128.0) /
                     (129.0 / 128.0) / (1.0 + 0x1p-29) * (1.0 - 0x1p-40);
    const double hi = floor(q / 0x1p64);
    if (hi >= 0x1p64) {                 // beyond 128 bits (bf16 counts above any in use)
      t.hi[P] = t.lo[P] = ~0ull;
      continue;
    }
    t.hi[P] = static_cast<unsigned long long>(hi);
    t.lo[P] = static_cast<unsigned long long>(q - hi * 0x1p64);
  }
  return t;
}

namespace {

// One block.  With a = the largest row-norm bound of the band's rows of A and
// b = that of B's rows (units of 2^norm_shift), every output of the band has
// |S| <= sqrt(a b) 2^shift (Cauchy-Schwarz).  The band takes the fewest moduli
// P in [least, most] with a b below the threshold t[P] (moduli_thresholds);
// the static count `most` covers every input.
// No shared memory: a kernel that needs some cannot start on an SM whose
// shared memory is configured for a running tensor-core GEMM, so this one
// would wait for the GEMM to end.  The warps meet through atomicMax on two
// zeroed slots (maxima[0..1]) instead.
constexpr int kModuliThreads = 512;
constexpr int kModuliUnroll = 4;

__device__ __forceinline__ unsigned long long max_of_rows(const unsigned long long* v, int64_t n) {
  unsigned long long m[kModuliUnroll] = {};
  for (int64_t i = threadIdx.x; i < n; i += int64_t(kModuliUnroll) * kModuliThreads) {
#pragma unroll
    for (int u = 0; u < kModuliUnroll; ++u) {
      const int64_t k = i + int64_t(u) * kModuliThreads;
      if (k < n) m[u] = max(m[u], __ldcg(v + k));       // all loads of a step in flight
    }
  }
#pragma unroll
  for (int u = 1; u < kModuliUnroll; ++u) m[0] = max(m[0], m[u]);
#pragma unroll
  for (int w = 16; w >= 1; w /= 2) m[0] = max(m[0], __shfl_xor_sync(0xFFFFFFFFu, m[0], w));
  return m[0];
}

// Smallest, over the 64-row blocks of `rows` rows, of the block's largest
// deep count (one warp per block in turn; the warp's lanes hold the result).
__device__ __forceinline__ unsigned min_block_max(const int* count, int64_t rows) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned mn = ~0u;
  for (int64_t blk = warp; blk * kTile < rows; blk += kModuliThreads / 32) {
    int mx = 0;
#pragma unroll
    for (int h = 0; h < kTile / 32; ++h) {
      const int64_t i = blk * kTile + lane + 32 * h;
      if (i < rows) mx = max(mx, __ldcg(count + i));
    }
    mn = min(mn, static_cast<unsigned>(__reduce_max_sync(0xFFFFFFFFu, mx)));
  }
  return mn;
}

__global__ void __launch_bounds__(kModuliThreads) moduli_kernel(
    const unsigned long long* normA, int64_t rowsA, const unsigned long long* normB, int64_t rowsB,
    int least, int most, int* used, int band, unsigned long long* maxima, ModuliThresholds thr,
    const int* countA, const int* countB, int cap) {
  const unsigned long long a_w = max_of_rows(normA, rowsA);
  const unsigned long long b_w = max_of_rows(normB, rowsB);
  unsigned mnA = ~0u, mnB = ~0u;
  if (countA != nullptr) {
    mnA = min_block_max(countA, rowsA);
    mnB = min_block_max(countB, rowsB);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicMax(maxima, a_w);
    atomicMax(maxima + 1, b_w);
    // minima through atomicMax of the complements on the zeroed slots 2, 3
    atomicMax(maxima + 2, static_cast<unsigned long long>(~mnA));
    atomicMax(maxima + 3, static_cast<unsigned long long>(~mnB));
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  const unsigned long long a = atomicAdd(maxima, 0ull);        // read at L2, after every warp
  const unsigned long long b = atomicAdd(maxima + 1, 0ull);
  int P = choose_moduli(a, b, least, most, thr);
  if (countA != nullptr && rowsA > 0 && rowsB > 0) {
    const unsigned minA = ~static_cast<unsigned>(atomicAdd(maxima + 2, 0ull));
    const unsigned minB = ~static_cast<unsigned>(atomicAdd(maxima + 3, 0ull));
    if (static_cast<uint64_t>(minA) + minB > static_cast<uint64_t>(cap)) P = 0;
  }
  *used = P;
  if (band >= 0 && band < kModuliRecord) g_moduli_record[band] = P;
}

}  // namespace

cudaError_t launch_moduli(const unsigned long long* normA, int64_t rowsA,
                          const unsigned long long* normB, int64_t rowsB, int bf16, int least,
                          int most, int* used, int band, unsigned long long* maxima,
                          const int* countA, const int* countB, int cap, cudaStream_t stream) {
  moduli_kernel<<<1, kModuliThreads, 0, stream>>>(normA, rowsA, normB, rowsB, least, most, used,
                                                  band, maxima, moduli_thresholds(bf16), countA,
                                                  countB, cap);
  note_launch();
  return cudaGetLastError();
}

bool fused_residues_ok(const ResidueOperand& o, int bf16) {
  return o.K <= kFusedK && rows_layout(o, bf16);
}

cudaError_t launch_residues_fused(const ResidueOperand& o0, const ResidueOperand* o1, int bf16,
                                  int nplanes, const FusedBand& fb, cudaStream_t stream) {
  const int64_t b0 = plane_rows(o0.rows), b1 = o1 != nullptr ? plane_rows(o1->rows) : 0;
  if (b0 + b1 == 0 || b0 + b1 > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(b0 + b1));
  const ResidueOperand& second = o1 != nullptr ? *o1 : o0;
  const bool grouped = o0.group_rows > 0 || second.group_rows > 0;
  const cudaError_t e = with_planes(bf16, nplanes, [&](auto B, auto P) {
    constexpr int kB = decltype(B)::value, kP = decltype(P)::value;
    if (grouped)
      residue_fused_kernel<kB, kP, true><<<grid, kThreads, 0, stream>>>(o0, second, static_cast<unsigned>(b0), fb);
    else
      residue_fused_kernel<kB, kP, false><<<grid, kThreads, 0, stream>>>(o0, second, static_cast<unsigned>(b0), fb);
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

namespace {
std::atomic<int> g_moduli_bands{0};
}  // namespace

void note_moduli_bands(int bands) { g_moduli_bands.store(bands, std::memory_order_relaxed); }

int moduli_record(int* out, int max) {
  int rec[kModuliRecord];
  if (cudaMemcpyFromSymbol(rec, g_moduli_record, sizeof(rec)) != cudaSuccess) return -1;
  int n = g_moduli_bands.load(std::memory_order_relaxed);
  n = n < kModuliRecord ? n : kModuliRecord;
  n = n < max ? n : max;
  for (int i = 0; i < n && out != nullptr; ++i) out[i] = rec[i];
  return n;
}

namespace {


// one launch over o0's row blocks, then o1's (both of the same layout)
cudaError_t residues_launch(const ResidueOperand& o0, const ResidueOperand& o1, int64_t blocks0,
                            int64_t blocks1, bool rows, int bf16, int nplanes, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>((o0.Kp + kTileK - 1) / kTileK), static_cast<unsigned>(blocks0 + blocks1));
  const unsigned split = static_cast<unsigned>(blocks0);
  const cudaError_t e = with_planes(bf16, nplanes, [&](auto B, auto P) {
    if (rows)
      residue_rows_kernel<decltype(B)::value, decltype(P)::value><<<grid, kThreads, 0, stream>>>(o0, o1, split);
    else {
      // its shared-memory tile must not keep it off SMs whose shared memory a
      // running tensor-core GEMM has configured for itself: with the default
      // carveout a later band's planes waited for the GEMM to end (DetLinear
      // wgrad 842 -> 831 us with the largest carveout preferred)
      static PerDeviceOnce carveout;             // the attribute is per device
      carveout.run([](int) {
        cudaFuncSetAttribute(residue_kernel<decltype(B)::value, decltype(P)::value>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        cudaGetLastError();                      // a preference only: never the caller's error
        return cudaSuccess;
      });
      residue_kernel<decltype(B)::value, decltype(P)::value><<<grid, kThreads, 0, stream>>>(o0, o1, split);
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_residues(const ResidueOperand& o, int bf16, int nplanes, cudaStream_t stream) {
  if (o.rows == 0 || o.Kp == 0) return cudaSuccess;
  return residues_launch(o, o, (o.rows + kTileRows - 1) / kTileRows, 0, rows_layout(o, bf16), bf16,
                         nplanes, stream);
}

cudaError_t launch_residues2(const ResidueOperand& o0, const ResidueOperand& o1, int bf16, int nplanes,
                             cudaStream_t stream) {
  const bool r0 = rows_layout(o0, bf16), r1 = rows_layout(o1, bf16);
  if (o0.rows == 0 || o1.rows == 0 || r0 != r1 || o0.Kp != o1.Kp) {
    cudaError_t e = launch_residues(o0, bf16, nplanes, stream);
    return e == cudaSuccess ? launch_residues(o1, bf16, nplanes, stream) : e;
  }
  if (o0.Kp == 0) return cudaSuccess;
  return residues_launch(o0, o1, (o0.rows + kTileRows - 1) / kTileRows,
                         (o1.rows + kTileRows - 1) / kTileRows, r0, bf16, nplanes, stream);
}

// Every copy of the bulk write-out starts 16-byte aligned: residue rows and
// digit rows (N a multiple of 16) and both bases.
bool partial_bulk_ok(const GemmArgs& g, const ReconArgs& ra) {
  return g.P != nullptr && (g.N % 16) == 0 && (reinterpret_cast<uintptr_t>(ra.res) % 16) == 0 &&
         (reinterpret_cast<uintptr_t>(g.P) % 16) == 0;
}

cudaError_t launch_reconstruct_fast(const GemmArgs& g, const ReconArgs& ra, cudaStream_t stream) {
  const int64_t band = ra.m_end - ra.m_begin;
  if (g.M * g.N == 0 || band <= 0) return cudaSuccess;
  cudaError_t e;
  if (g.P != nullptr) {
    // each block walks several rows, two at a time (measured at 4096 x 4096:
    // 512 blocks per column of blocks beat one row per block by 3 %)
    dim3 pgrid(static_cast<unsigned>((g.N + kThreads - 1) / kThreads),
               static_cast<unsigned>(band < 512 ? band : 512));
    // bulk copies where every row of residues and of digits starts 16-byte aligned
    const bool bulk = partial_bulk_ok(g, ra);
    if (bulk) {                                   // five blocks per SM, each a chunk of rows
      int dev = 0, sms = 0;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      pgrid.x = static_cast<unsigned>((g.N + kBulkCols - 1) / kBulkCols);
      const int64_t per_col =
          (int64_t(sms > 0 ? sms : 1) * kBulkBlocksPerSm + pgrid.x - 1) / pgrid.x;
      pgrid.y = static_cast<unsigned>(band < per_col ? band : per_col);
    }
    e = with_planes(g.bf16, ra.nplanes, [&](auto B, auto P) {
      constexpr int kB = decltype(B)::value, kP = decltype(P)::value;
      if (bulk) {
        static PerDeviceOnce carveout;            // five 43 KB blocks per SM
        carveout.run([](int) {
          cudaFuncSetAttribute(partial_bulk_kernel<kB, kP>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
          cudaGetLastError();
          return cudaSuccess;
        });
        partial_bulk_kernel<kB, kP><<<pgrid, kBulkCols, 0, stream>>>(g, ra);
      } else {
        partial_fast_kernel<kB, kP><<<pgrid, kThreads, 0, stream>>>(g, ra);
      }
      return cudaSuccess;
    });
  } else {
    const int64_t cols_per_block = int64_t(kThreads) * kReconCols;
    // blocks walk several rows, two per step (1024 per column of blocks)
    dim3 grid(static_cast<unsigned>((g.N + cols_per_block - 1) / cols_per_block),
              static_cast<unsigned>(band < 1024 ? band : 1024));
    e = with_planes(g.bf16, ra.nplanes, [&](auto B, auto P) {
      constexpr int kB = decltype(B)::value, kP = decltype(P)::value;
      if (g.batch > 1) reconstruct_fast_kernel<kB, kP, true><<<grid, kThreads, 0, stream>>>(g, ra);
      else reconstruct_fast_kernel<kB, kP, false><<<grid, kThreads, 0, stream>>>(g, ra);
      return cudaSuccess;
    });
  }
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_reconstruct_deep(const GemmArgs& g, const ReconArgs& ra, int* deep_lists,
                                    int* deep_counters, int parts, int blocks_per_sm,
                                    cudaStream_t stream) {
  const int64_t band = ra.m_end - ra.m_begin;
  if (g.M * g.N == 0 || band <= 0 || (parts & (kDeepRows | kDeepCols)) == 0) return cudaSuccess;
  // deep rows and columns: index lists [M] and [N] and their two counters,
  // filled by the routing step.  The kernel waits on memory most of the
  // time; one block per SM leaves room for the fast kernel beside it.
  const int* rows = deep_lists;
  const int* cols = deep_lists + g.M;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const unsigned dgrid = static_cast<unsigned>((sms > 0 ? sms : 1) * (blocks_per_sm > 1 ? 2 : 1));
  const cudaError_t e = with_planes(g.bf16, ra.nplanes, [&](auto B, auto P) {
    reconstruct_deep_kernel<decltype(B)::value, decltype(P)::value>
        <<<dgrid, kThreads, 0, stream>>>(g, ra, rows, cols, deep_counters, parts);
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

}  // namespace det
