// Device arithmetic of the exact-sum GEMM: operand decode, digit
// normalisation and the single round-to-nearest-even to binary32.
//
// det-train page, section "Method": products are exact, their base-2^32
// limbs are added into signed int64 digits, and the final digits are
// carry-normalised and rounded once.  Everything here is integer arithmetic
// written from the IEEE-754 binary32 definition; no floating-point
// instruction touches a value on this path.
#pragma once

#include <stdint.h>

namespace det {

constexpr int kDigits = 18;      // radix-2^32 digits per output
constexpr int kPlanes = 20;      // + product count + non-finite count
constexpr int kLsbBias = 298;    // digit 0 weighs 2^-298
constexpr uint32_t kNanBits = 0x7FC00000u;

// ---------------------------------------------------------------------------
// Operand decode.  A finite binary32 x is (-1)^s * m * 2^e with an integer
// significand m < 2^24 and e the weight of its last significand bit:
// normal: m = 1.fraction (24 bits), e = biased - 150; subnormal or zero:
// m = fraction, e = -149.  bf16 is the top half of a binary32 pattern.
// ---------------------------------------------------------------------------
struct Decoded {
  int32_t m;        // signed significand, |m| < 2^24 (0 for zero / non-finite)
  int32_t e;        // exponent of the significand's last bit, in [-149, 104]
  bool nonfinite;
};

__device__ __forceinline__ Decoded decode_f32_bits(uint32_t bits) {
  uint32_t biased = (bits >> 23) & 0xFFu;
  uint32_t frac = bits & 0x7FFFFFu;
  Decoded d;
  d.nonfinite = biased == 0xFFu;
  uint32_t mag = frac | (biased != 0 ? 0x800000u : 0u);
  mag = d.nonfinite ? 0u : mag;
  d.m = (bits >> 31) ? -static_cast<int32_t>(mag) : static_cast<int32_t>(mag);
  d.e = static_cast<int32_t>(biased > 1u ? biased : 1u) - 150;
  if (d.nonfinite) d.e = 0;
  return d;
}

// Exponent key of a binary32 pattern (a bf16 widened to binary32): the
// biased exponent, with subnormals counted as 1 (their last-bit exponent,
// -149, is that of biased exponent 1), and 0 for zero and non-finite values.
// For a live element, key - 150 is the exponent e of its last significand bit.
__device__ __forceinline__ int exp_key(uint32_t bits) {
  const uint32_t a = bits & 0x7FFFFFFFu;
  const int key = max(static_cast<int>(a >> 23), 1);
  return (a == 0u || a >= 0x7F800000u) ? 0 : key;
}

template <int kBf16>
__device__ __forceinline__ uint32_t load_bits(const void* base, int64_t idx) {
  if (kBf16) {
    uint16_t h = __ldg(static_cast<const unsigned short*>(base) + idx);
    return static_cast<uint32_t>(h) << 16;
  } else {
    return __ldg(static_cast<const unsigned int*>(base) + idx);
  }
}

// ---------------------------------------------------------------------------
// Carry normalisation: arbitrary int64 digits (|d| < 2^62) -> 17 unsigned
// 32-bit words plus a signed top digit.  The value is unchanged:
//   sum_j d[j] 2^(32j)  ==  sum_{j<17} w[j] 2^(32j) + top * 2^(32*17).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void normalise_digits(const int64_t (&d)[kDigits], uint32_t (&w)[kDigits - 1],
                                                 int64_t& top) {
  int64_t carry = 0;
#pragma unroll
  for (int j = 0; j < kDigits - 1; ++j) {
    int64_t v = d[j] + carry;
    w[j] = static_cast<uint32_t>(v);
    carry = v >> 32;                  // arithmetic shift: floor division by 2^32
  }
  top = d[kDigits - 1] + carry;
}

// ---------------------------------------------------------------------------
// Round once to binary32, ties to even.  Input: the exact value as
// sum_{j<17} w[j] 2^(32j) + top 2^544, in units of 2^-298, two's complement
// through `top`.  Output: the binary32 bit pattern.
//   exact zero -> +0; nonzero values that round to zero keep their sign;
//   values that round to 2^128 or beyond -> +-inf.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t round_to_f32_bits(const uint32_t (&w)[kDigits - 1], int64_t top) {
  const bool neg = top < 0;
  // One pass over the words of the magnitude (negated on the fly when the
  // value is negative: magnitude = ~x + 1), keeping only registers: the
  // leading nonzero word, the two words below it, and the OR of all lower ones.
  uint32_t carry = neg ? 1u : 0u;
  uint32_t p1 = 0, p2 = 0, older = 0;              // the two previous words, OR of the rest
  uint32_t whi = 0, wmid = 0, wlo = 0, rest = 0;    // 96-bit window below the leading bit
  int hi = -1;                                      // index of the leading nonzero word
#pragma unroll
  for (int j = 0; j < kDigits - 1; ++j) {
    uint32_t v = w[j];
    if (neg) {
      v = ~v + carry;
      carry = (carry != 0u && v == 0u) ? 1u : 0u;
    }
    if (v != 0u) {
      whi = v;
      wmid = p1;
      wlo = p2;
      rest = older;
      hi = j;
    }
    older |= p2;
    p2 = p1;
    p1 = v;
  }
  const uint64_t mag_top = neg ? static_cast<uint64_t>(~top) + carry : static_cast<uint64_t>(top);
  const uint32_t sign = neg ? 0x80000000u : 0u;
  if (mag_top != 0) return sign | 0x7F800000u;     // >= 2^(544-298): overflow
  if (hi < 0) return 0u;                            // exact zero -> +0
  const int msb = 32 * hi + 31 - __clz(whi);        // bit index of the leading 1
  if (msb >= 128 + kLsbBias) return sign | 0x7F800000u;   // |x| >= 2^128

  // ulp bit index: 23 bits below the leading one, but never below 2^-149
  const int s = max(msb - 23, kLsbBias - 149);
  const int sh = s - 32 * (hi - 2);                 // ulp position inside the window, >= 41
  const unsigned __int128 win = (static_cast<unsigned __int128>(whi) << 64) |
                                (static_cast<unsigned __int128>(wmid) << 32) | wlo;
  uint64_t q = sh < 96 ? static_cast<uint64_t>(win >> sh) : 0u;
  const uint32_t half = (sh - 1) < 96 ? static_cast<uint32_t>(win >> (sh - 1)) & 1u : 0u;
  const unsigned __int128 below =
      (sh - 1) < 96 ? (win & ((static_cast<unsigned __int128>(1) << (sh - 1)) - 1)) : win;
  const bool sticky = (below != 0) || (rest != 0u);
  if (half && (sticky || (q & 1u))) ++q;
  int qexp = s - kLsbBias;                          // exponent of one ulp
  if (q == (1ull << 24)) {
    q >>= 1;
    ++qexp;
  }
  if (qexp > 104) return sign | 0x7F800000u;        // rounded up to 2^128
  uint32_t bits;
  if (q >= (1ull << 23)) {
    bits = (static_cast<uint32_t>(qexp + 150) << 23) | static_cast<uint32_t>(q - (1ull << 23));
  } else {
    bits = static_cast<uint32_t>(q);                // subnormal (qexp == -149) or zero
  }
  return sign | bits;
}

// The binary32 pattern of a 64-bit integer t in [2^63, 2^64), rounded to
// nearest even, in 32-bit integer steps (a 64-bit integer-to-float
// conversion would run on the narrow fp64 pipe): bits 63..40 are the
// significand, bit 39 the rounding bit, bits 38..0 the sticky bits.  The
// exponent field is 190 (2^63); a significand that rounds up to 2^24 carries
// into it.
__host__ __device__ __forceinline__ uint32_t f32_bits_of_top(uint64_t t) {
  const uint32_t t_hi = static_cast<uint32_t>(t >> 32), t_lo = static_cast<uint32_t>(t);
  const uint32_t mant = t_hi >> 8;                                  // in [2^23, 2^24)
  const uint32_t sticky = ((t_hi & 0x7Fu) | t_lo) != 0u ? 1u : 0u;
  const uint32_t up = (t_hi >> 7) & (sticky | mant) & 1u;
  return (189u << 23) + mant + up;
}

}  // namespace det
