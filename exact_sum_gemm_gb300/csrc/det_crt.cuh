// The CRT as one sum of products, with compile-time constants for each count
// of moduli (used by the reconstruction kernels).
#pragma once

#include <stdint.h>

#include "det_residue.cuh"

namespace det {

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
template <int P, int i, bool kTop>
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
    if constexpr (kTop) acc3 += r[i] * c3;
    Q += r[i] * w;
    crt_terms<P, i + 1, kTop>(r, acc, acc3, Q);
  }
}

// Whether |S| < M / 2 fits a 96-bit two's-complement value (M < 2^95), so
// that the sum modulo 2^96 -- three limbs -- determines it: the first 12
// moduli (M < 2^94.6, every f32 band at the least count) and every bf16 count.
__host__ __device__ constexpr bool crt_three_limbs(int P) {
  double m = 1.0;
  for (int i = 0; i < P; ++i) m *= static_cast<double>(modulus(i));
  return m < 0x1p95;
}

// S (two's complement, hi:lo) from the balanced residues r_0 .. r_{P-1}
// (|r_i| <= (p_i - 1)/2), given |S| < M / (2 (1 + 2^-7)), the margin that
// residue_planes_needed keeps.  Q / 2^20 is within 14 * 127 / 2^21 < 2^-10
// of S'/M = q + S/M, and |S/M| < 1/2 - 2^-8.01, so Q rounds to q.
template <int P>
__host__ __device__ __forceinline__ void crt_s128(const int32_t (&r)[kNumModuli], uint64_t& lo,
                                                  uint64_t& hi) {
  static_assert(P >= 1 && P <= kNumModuli, "moduli in use");
  constexpr bool kTop = !crt_three_limbs(P);
  int64_t acc[3] = {0, 0, 0};
  int32_t acc3 = 0, Q = 0;                         // |Q| < 14 * 127 * 2^19 < 2^30
  crt_terms<P, 0, kTop>(r, acc, acc3, Q);
  const int32_t q = (Q + (1 << (kCrtWeightBits - 1))) >> kCrtWeightBits;
  static_assert(crt_negM_limb(P, 3) < (1 << 14) && crt_negM_limb(P, 3) > -(1 << 14), "top limb");
  acc[0] += static_cast<int64_t>(q) * crt_negM_limb(P, 0);
  acc[1] += static_cast<int64_t>(q) * crt_negM_limb(P, 1);
  acc[2] += static_cast<int64_t>(q) * crt_negM_limb(P, 2);
  if constexpr (kTop) acc3 += q * crt_negM_limb(P, 3);
  // S = acc0 + acc1 2^32 + acc2 2^64 (+ acc3 2^96) modulo 2^128 (2^96 with
  // three limbs); |acc_l| < 2^43
  const uint64_t a0 = static_cast<uint64_t>(acc[0]);
  const uint64_t a1lo = static_cast<uint64_t>(acc[1]) << 32;
  lo = a0 + a1lo;
  const uint64_t carry = lo < a0 ? 1u : 0u;
  hi = static_cast<uint64_t>(acc[0] >> 63) + static_cast<uint64_t>(acc[1] >> 32) + carry +
       static_cast<uint64_t>(acc[2]);
  if constexpr (kTop) {
    hi += static_cast<uint64_t>(static_cast<uint32_t>(acc3)) << 32;
  } else {
    // S modulo 2^96, sign-extended from bit 95
    hi = static_cast<uint64_t>(static_cast<int64_t>(hi << 32) >> 32);
  }
}

}  // namespace det
