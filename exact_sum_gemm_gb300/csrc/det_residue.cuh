// Moduli and launch plumbing of the residue (CRT) decomposition.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "det_kernels.h"

namespace det {

// Odd, pairwise coprime moduli in [197, 255].  The operand planes hold
// residues r with |r| <= 138 (nearly balanced, exact in bf16, which holds
// integers up to 256), so a product of two is at most 138^2 = 19044 in
// magnitude, and 832 such products plus a reduced carry (< 131) stay below
// 2^24, where fp32 accumulation is exact.  The product of all 14 moduli
// exceeds 2^109, enough for |S| < 2^19 * 2^86 * 2 (f32 shallow integers are
// below 2^(24+19)).
constexpr int kNumModuli = 14;
__host__ __device__ constexpr int modulus(int i) {
  return i == 0 ? 255 : i == 1 ? 253 : i == 2 ? 251 : i == 3 ? 247 : i == 4 ? 241 : i == 5 ? 239
       : i == 6 ? 233 : i == 7 ? 229 : i == 8 ? 227 : i == 9 ? 223 : i == 10 ? 217 : i == 11 ? 211
       : i == 12 ? 199 : 197;
}
// Balanced representatives, inverses and products modulo the moduli (compile
// time).
__host__ __device__ constexpr int balanced_rep(long long x, int p) {
  long long r = x % p;
  if (r < 0) r += p;
  return static_cast<int>(r > (p - 1) / 2 ? r - p : r);
}
__host__ __device__ constexpr int inverse_mod(int a, int p) {
  for (int c = 1; c < p; ++c)
    if ((a * c) % p == 1) return c;
  return 0;
}
// The CRT as one sum.  For the first P moduli, with M = p_0 ... p_{P-1}, the
// balanced residues r_i of an integer S with |S| < M/2 give
//   S = sum_i r_i C_i - q M,   C_i = (M / p_i) c_i,  c_i = (M / p_i)^-1 mod p_i,
// q = the integer nearest to sum_i r_i c_i / p_i (that sum is S'/M for
// S' = sum_i r_i C_i, and S'/M - q = S/M).  The reconstruction estimates q in
// fixed point, Q = sum_i r_i W_i with W_i = round(2^20 c_i / p_i), and sums
// the products modulo 2^128 in four signed 32-bit limbs (value = sum_l
// L_l 2^(32 l)), so every limb sum is an exact 64-bit integer.  These are the
// compile-time constants; c_i is taken balanced, so |c_i / p_i| < 1/2.
__host__ __device__ constexpr int crt_c(int P, int i) {
  int r = 1;                                   // (M / p_i) mod p_i
  for (int j = 0; j < P; ++j)
    if (j != i) r = (r * (modulus(j) % modulus(i))) % modulus(i);
  return balanced_rep(inverse_mod(r, modulus(i)), modulus(i));
}
// limb l (0..3) of x mod 2^128, x = (product of the first P moduli except
// `skip`) * factor, as a signed limb (the limbs below carry into it)
__host__ __device__ constexpr int32_t crt_limb_of(int P, int skip, long long factor, int l) {
  unsigned long long w[4] = {1, 0, 0, 0};              // 32-bit limbs held in 64 bits
  for (int j = 0; j < P; ++j) {
    if (j == skip) continue;
    unsigned long long carry = 0;
    for (int t = 0; t < 4; ++t) {
      const unsigned long long v = w[t] * static_cast<unsigned long long>(modulus(j)) + carry;
      w[t] = v & 0xFFFFFFFFull;
      carry = v >> 32;
    }
  }
  const bool neg = factor < 0;
  const unsigned long long f = static_cast<unsigned long long>(neg ? -factor : factor);
  unsigned long long carry = 0;
  for (int t = 0; t < 4; ++t) {
    const unsigned long long v = w[t] * f + carry;
    w[t] = v & 0xFFFFFFFFull;
    carry = v >> 32;
  }
  if (neg) {                                            // two's complement modulo 2^128
    unsigned long long c = 1;
    for (int t = 0; t < 4; ++t) {
      const unsigned long long v = (~w[t] & 0xFFFFFFFFull) + c;
      w[t] = v & 0xFFFFFFFFull;
      c = v >> 32;
    }
  }
  long long borrow = 0;                                 // signed limbs in [-2^31, 2^31)
  int32_t out = 0;
  for (int t = 0; t <= l; ++t) {
    long long v = static_cast<long long>(w[t]) + borrow;
    borrow = 0;
    if (v >= (1ll << 31)) {
      v -= 1ll << 32;
      borrow = 1;
    }
    out = static_cast<int32_t>(v);
  }
  return out;
}
__host__ __device__ constexpr int32_t crt_C_limb(int P, int i, int l) {
  return crt_limb_of(P, i, crt_c(P, i), l);
}
__host__ __device__ constexpr int32_t crt_negM_limb(int P, int l) {
  return crt_limb_of(P, -1, -1, l);
}
__host__ __device__ constexpr int32_t crt_W(int P, int i) {
  // round(2^20 c / p) for |c| < p/2, exactly, in integers
  const long long num = static_cast<long long>(crt_c(P, i)) * (1ll << 21) + modulus(i);
  const long long den = 2ll * modulus(i);
  return static_cast<int32_t>(num >= 0 ? num / den : -((-num + den - 1) / den));
}
constexpr int kCrtWeightBits = 20;

// The top limb of every C_i and of -M is below 2^14 in magnitude (M < 2^110),
// so its sum stays within 32 bits: 14 * 127 * 2^14 + 2^10 * 2^14 < 2^25.
template <int P, int i>
__host__ __device__ __forceinline__ void crt_terms(const int32_t (&r)[kNumModuli], int64_t (&acc)[3],
                                                   int32_t& acc3, int32_t& Q) {
  if constexpr (i < P) {
    constexpr int32_t c0 = crt_C_limb(P, i, 0), c1 = crt_C_limb(P, i, 1);
    constexpr int32_t c2 = crt_C_limb(P, i, 2), c3 = crt_C_limb(P, i, 3);
    static_assert(c3 < (1 << 14) && c3 > -(1 << 14), "top limb below 2^14");
    constexpr int32_t w = crt_W(P, i);
#ifdef __CUDA_ARCH__
    // one 32 x 32 -> 64-bit signed multiply-add each
    asm("mad.wide.s32 %0, %1, %2, %0;" : "+l"(acc[0]) : "r"(r[i]), "n"(c0));
    asm("mad.wide.s32 %0, %1, %2, %0;" : "+l"(acc[1]) : "r"(r[i]), "n"(c1));
    asm("mad.wide.s32 %0, %1, %2, %0;" : "+l"(acc[2]) : "r"(r[i]), "n"(c2));
#else
    acc[0] += static_cast<int64_t>(r[i]) * c0;
    acc[1] += static_cast<int64_t>(r[i]) * c1;
    acc[2] += static_cast<int64_t>(r[i]) * c2;
#endif
    acc3 += r[i] * c3;
    Q += r[i] * w;
    crt_terms<P, i + 1>(r, acc, acc3, Q);
  }
}

// S (two's complement, hi:lo) from the balanced residues r_0 .. r_{P-1}
// (|r_i| <= (p_i - 1)/2), given |S| < M / (2 (1 + 2^-7)), the margin that
// residue_planes_needed keeps.  Q / 2^20 is within 14 * 127 / 2^21 < 2^-10
// of S'/M = q + S/M, and |S/M| < 1/2 - 2^-8.01, so Q rounds to q.
template <int P>
__host__ __device__ __forceinline__ void crt_s128(const int32_t (&r)[kNumModuli], uint64_t& lo,
                                                  uint64_t& hi) {
  static_assert(P >= 1 && P <= kNumModuli, "moduli in use");
  int64_t acc[3] = {0, 0, 0};
  int32_t acc3 = 0, Q = 0;                         // |Q| < 14 * 127 * 2^19 < 2^30
  crt_terms<P, 0>(r, acc, acc3, Q);
  const int32_t q = (Q + (1 << (kCrtWeightBits - 1))) >> kCrtWeightBits;
  static_assert(crt_negM_limb(P, 3) < (1 << 14) && crt_negM_limb(P, 3) > -(1 << 14), "top limb");
  acc[0] += static_cast<int64_t>(q) * crt_negM_limb(P, 0);
  acc[1] += static_cast<int64_t>(q) * crt_negM_limb(P, 1);
  acc[2] += static_cast<int64_t>(q) * crt_negM_limb(P, 2);
  acc3 += q * crt_negM_limb(P, 3);
  // S = acc0 + acc1 2^32 + acc2 2^64 + acc3 2^96 (mod 2^128); |acc_l| < 2^43
  const uint64_t a0 = static_cast<uint64_t>(acc[0]);
  const uint64_t a1lo = static_cast<uint64_t>(acc[1]) << 32;
  lo = a0 + a1lo;
  const uint64_t carry = lo < a0 ? 1u : 0u;
  hi = static_cast<uint64_t>(acc[0] >> 63) + static_cast<uint64_t>(acc[1] >> 32) + carry +
       static_cast<uint64_t>(acc[2]) + (static_cast<uint64_t>(static_cast<uint32_t>(acc3)) << 32);
}

// Exact modular reduction in binary32 (integers below 2^24 are exact there,
// and the fp32 FMA pipes outrun the integer multiplier).  For an integer-
// valued a with |a| <= 2^26 and an odd modulus p in [197, 255], with
// inv_p = 1/p to within one ulp (so |a * inv_p| < 2^19, where adding
// 1.5*2^23 rounds to an integer):
//   q = (a * inv_p + 1.5*2^23) - 1.5*2^23      (one rounding to an integer)
//   r = a - q * p                               (one fma: exact, r is small)
// Before rounding, q is within |a|/p * 2^-23 of the real a/p.  a/p is never
// a half-integer (p is odd) and a non-integer a/p lies at least 1/(2p) > 2^-9
// from one; so whenever |a| < 2^14 * p the rounding gives the nearest integer
// and r is the balanced residue in [-(p-1)/2, (p-1)/2].  Otherwise q may be
// one off: |r| <= p * (1/2 + |a|/p * 2^-23), which is below 131 for
// |a| <= 2^24 and below 139 for |a| <= 2^26.  A zero result is +0 unless a
// is -0.
constexpr float kRoundMagic = 12582912.0f;           // 1.5 * 2^23

__device__ __forceinline__ float near_mod_f32(float a, float p, float inv_p) {
  const float q = __fsub_rn(__fmaf_rn(a, inv_p, kRoundMagic), kRoundMagic);
  return __fmaf_rn(-q, p, a);
}

constexpr int kChunkK = 832;      // K per exact fp32 accumulation window (13 stages)
constexpr int kStageK = 64;       // K per TMA/MMA stage (one 128-byte swizzle row of bf16)
static_assert(kChunkK % kStageK == 0, "accumulation windows are whole stages");
static_assert(int64_t(kChunkK) * 138 * 138 + 131 < (int64_t(1) << 24), "window stays exact in fp32");

// Plane layout.  Rows are taken in groups of kPlaneRows; for each group and
// 64-k stage the nplanes planes follow one another, each a 32 x 64 bf16 block
// (4 KB, 128 bytes per row):
//   plane u of element (r, k) at
//   (((r / 32) * Kp/64 + k / 64) * nplanes + u) * 2048 + (r % 32) * 64 + k % 64.
// The residue kernel writes an element pair's planes at fixed 4 KB steps, and
// one modulus's stage for 32 rows is one contiguous 4 KB block for the TMA.
// Padding rows (up to a multiple of 32) hold zero residues.
constexpr int kPlaneRows = 32;
inline int64_t plane_rows(int64_t rows) { return (rows + kPlaneRows - 1) / kPlaneRows * kPlaneRows; }

struct ResidueOperand {
  const void* X;
  int64_t ld;
  int op;
  int64_t rows;
  int64_t K;
  int64_t Kp;                 // K rounded up to kStageK (zero padded)
  const int* emax;            // [rows]
  __nv_bfloat16* planes;      // [rows/32][Kp/64][nplanes][32][64] (rows padded to 32, see
                              // kPlaneRows)
  int* list_count;            // [rows], zeroed before the launch
  uint2* list;                // [rows][cap]: (k, raw bits) of deep / non-finite elements
  int cap;
};

struct ReconArgs {
  const int8_t* res;          // [nplanes][M][N] balanced residues, |r| <= (p_i - 1) / 2
  int nplanes;
  const int* emaxA;
  const int* emaxB;
  const uint8_t* route;       // 64x64 tiles: 1 = general kernel (skipped here)
  const int* countA;
  const uint2* listA;
  const int* countB;
  const uint2* listB;
  int cap;
  const int* error;           // nonzero: the tensor-core kernel gave up (outputs NaN)
  int64_t m_begin, m_end;     // rows of C handled by this launch (a band)
};

int residue_planes_needed(const GemmArgs& g);
cudaError_t launch_residues(const ResidueOperand& o, int bf16, int nplanes, cudaStream_t stream);
// Two operands' planes in one launch (one grid covering both).
cudaError_t launch_residues2(const ResidueOperand& o0, const ResidueOperand& o1, int bf16, int nplanes,
                             cudaStream_t stream);
// The outputs of a band whose row of A and column of B hold no deep element.
cudaError_t launch_reconstruct_fast(const GemmArgs& g, const ReconArgs& ra, cudaStream_t stream);
// The band's other outputs (independent of the fast kernel: both may run at
// once).  deep_lists: the rows of A then the columns of C that hold deep
// elements (M + N ints), with their two counts in deep_counters, as the
// routing step lists them.
cudaError_t launch_reconstruct_deep(const GemmArgs& g, const ReconArgs& ra, int* deep_lists,
                                    int* deep_counters, cudaStream_t stream);

struct ResGemmArgs {
  const __nv_bfloat16* A;     // [M/32][Kp/64][nplanes][32][64] (ResidueOperand::planes)
  const __nv_bfloat16* B;     // [N/32][Kp/64][nplanes][32][64]
  int64_t M, N, Kp;
  int nplanes;
  int8_t* res;                // [nplanes][.][N] balanced residues: plane u of row m at
  int64_t res_plane;          //   res + u * res_plane + m * N
  int* error;
};
cudaError_t launch_residue_gemm(const ResGemmArgs& a, cudaStream_t stream);
// The same GEMM with 256 x 256 tiles over CTA pairs (cta_group::2); returns
// cudaErrorNotSupported (nothing enqueued) where clusters of two cannot run.
cudaError_t launch_residue_gemm_pair(const ResGemmArgs& a, cudaStream_t stream);

}  // namespace det
