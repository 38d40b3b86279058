// Exact-sum GEMM oracle.  TEST INFRASTRUCTURE ONLY: nothing on the product
// path may include, link or call this file.  Only the test suite, the smoke
// check and the benchmark's CPU-baseline leg use it.
//
// What it computes (det-train page, section "Method"): every output of a
// bf16/f32 GEMM is the exact real sum of the exact fp64 products of its
// inputs, rounded a single time to binary32 with round-to-nearest,
// ties-to-even.  The section "Correctness" states the same property of the
// results.
//
// This is the plain definition written out, deliberately on a different
// route from the GPU kernels:
//   * operands are converted with ordinary C casts (float -> double), never
//     by bit decoding;
//   * each product is formed as one double multiply (24x24 significand bits
//     fit in 53, and the exponent range of a product of two binary32 values
//     lies well inside binary64, so the multiply is exact);
//   * the product is split with std::frexp into an integer significand and a
//     binary exponent;
//   * it is added into a FULLY NORMALISED two's-complement big integer
//     (32-bit words, carry propagated immediately), whose bit 0 weighs 2^-298,
//     the smallest nonzero |product| of two binary32 subnormals;
//   * the sum is rounded once, by the IEEE-754 binary32 rule written from its
//     definition (gradual underflow, overflow to +-inf).
//
// Readings where the pages are silent (each is also listed in the design
// notes of the repository):
//   * an exact zero sum is +0.0f; a nonzero sum that rounds to zero keeps its
//     sign;
//   * a product with a non-finite operand is not accumulated; it is counted,
//     and any output with a nonzero count is the canonical NaN 0x7FC00000;
//   * the canonical digit form of a sum is 18 digits of radix 2^32, digit j
//     weighing 2^(32j-298); digits 0..16 lie in [0, 2^32) and digit 17 carries
//     the sign.  (The pages fix only signed int64 digits of radix 2^32
//     covering the whole range of fp32 product exponents.)
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -shared -fPIC -pthread.
// Rows of the output are spread over std::threads; nothing else is clever.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr int kWords = 20;          // 640 bits of two's complement
constexpr int kLsbExp = -298;       // weight of bit 0 is 2^-298
constexpr int kDigits = 18;         // canonical digit count (radix 2^32)
constexpr int kPlanes = 20;         // digits, product count, non-finite count

struct Big {
  uint32_t w[kWords];
};

void big_zero(Big& b) { std::memset(b.w, 0, sizeof(b.w)); }

// b += mag * 2^pos   (mag < 2^64, 0 <= pos, pos + 64 < 640)
void big_add(Big& b, uint64_t mag, int pos) {
  int wi = pos / 32;
  int sh = pos % 32;
  unsigned __int128 v = static_cast<unsigned __int128>(mag) << sh;
  uint64_t carry = 0;
  for (int i = wi; i < kWords; ++i) {
    int rel = i - wi;
    uint64_t addend = rel < 3 ? static_cast<uint32_t>(v >> (32 * rel)) : 0u;
    uint64_t s = static_cast<uint64_t>(b.w[i]) + addend + carry;
    b.w[i] = static_cast<uint32_t>(s);
    carry = s >> 32;
    if (rel >= 2 && carry == 0) break;
  }
}

// b -= mag * 2^pos
void big_sub(Big& b, uint64_t mag, int pos) {
  int wi = pos / 32;
  int sh = pos % 32;
  unsigned __int128 v = static_cast<unsigned __int128>(mag) << sh;
  uint64_t borrow = 0;
  for (int i = wi; i < kWords; ++i) {
    int rel = i - wi;
    uint64_t sub = rel < 3 ? static_cast<uint32_t>(v >> (32 * rel)) : 0u;
    uint64_t cur = b.w[i];
    uint64_t need = sub + borrow;
    if (cur >= need) {
      b.w[i] = static_cast<uint32_t>(cur - need);
      borrow = 0;
    } else {
      b.w[i] = static_cast<uint32_t>(cur + (uint64_t(1) << 32) - need);
      borrow = 1;
    }
    if (rel >= 2 && borrow == 0) break;
  }
}

bool big_is_negative(const Big& b) { return (b.w[kWords - 1] >> 31) != 0; }

void big_negate(Big& b) {
  uint64_t carry = 1;
  for (int i = 0; i < kWords; ++i) {
    uint64_t s = static_cast<uint64_t>(~b.w[i]) + carry;
    b.w[i] = static_cast<uint32_t>(s);
    carry = s >> 32;
  }
}

int big_bit(const Big& b, int i) { return (b.w[i / 32] >> (i % 32)) & 1; }

// Add one exact product (a double holding an exact value that is a multiple
// of 2^-298) into the accumulator.
void add_exact_double(Big& acc, double p) {
  if (p == 0.0) return;
  int ex = 0;
  double f = std::frexp(std::fabs(p), &ex);            // |p| = f * 2^ex, f in [0.5, 1)
  uint64_t mant = static_cast<uint64_t>(std::ldexp(f, 53));  // exact, < 2^53
  int pos = ex - 53 - kLsbExp;                          // bit position of mant's LSB
  while (pos < 0) {                                     // value is a multiple of 2^-298
    mant >>= 1;                                         // so these bits are zero
    ++pos;
  }
  if (p > 0) big_add(acc, mant, pos);
  else big_sub(acc, mant, pos);
}

// Round a big integer (units of 2^-298) once to binary32, ties to even.
float big_round_to_f32(Big x) {
  bool neg = big_is_negative(x);
  if (neg) big_negate(x);
  int msb = -1;
  for (int i = kWords * 32 - 1; i >= 0; --i) {
    if (big_bit(x, i)) { msb = i; break; }
  }
  if (msb < 0) return 0.0f;                            // exact zero -> +0
  int e_msb = msb + kLsbExp;                           // exponent of the leading bit
  int q_exp = std::max(e_msb - 23, -149);              // exponent of one unit in the last place
  int s = q_exp - kLsbExp;                             // its bit index (>= 149)
  uint64_t q = 0;
  for (int i = msb; i >= s; --i) q = (q << 1) | static_cast<uint64_t>(big_bit(x, i));
  int half = big_bit(x, s - 1);
  int sticky = 0;
  for (int i = s - 2; i >= 0 && !sticky; --i) sticky = big_bit(x, i);
  if (half && (sticky || (q & 1))) ++q;
  if (q == (uint64_t(1) << 24)) {
    q >>= 1;
    ++q_exp;
  }
  float r;
  if (q_exp > 104) r = INFINITY;                       // q * 2^q_exp >= 2^128
  else r = static_cast<float>(std::ldexp(static_cast<double>(q), q_exp));  // exact
  return neg ? -r : r;
}

// Canonical digits: 0..16 in [0, 2^32), 17 signed (sign-extended top).
void big_to_digits(const Big& x, int64_t* d, int64_t stride) {
  for (int j = 0; j < kDigits - 1; ++j) d[j * stride] = static_cast<int64_t>(x.w[j]);
  // digit 17 is the signed value of words 17..19 (it fits int64 for every
  // sum the library can form: |value| < 2^575 units)
  int64_t top = static_cast<int64_t>(static_cast<int32_t>(x.w[kWords - 1]));
  top = top * (int64_t(1) << 32) + static_cast<int64_t>(x.w[kWords - 2]);
  int64_t w17 = static_cast<int64_t>(x.w[kDigits - 1]);
  d[(kDigits - 1) * stride] = top * (int64_t(1) << 32) + w17;
}

float load_elem(int dtype, const void* base, int64_t idx) {
  if (dtype == 0) {
    return static_cast<const float*>(base)[idx];
  }
  uint16_t h = static_cast<const uint16_t*>(base)[idx];
  uint32_t bits = static_cast<uint32_t>(h) << 16;      // bf16 is the top half of a binary32
  float f;
  std::memcpy(&f, &bits, sizeof(f));
  return f;
}

struct GemmArgs {
  int dtype;
  int64_t M, N, K;
  const void* A;
  int64_t sAm, sAk;
  const void* B;
  int64_t sBn, sBk;
  float* C;
  int64_t ldc;
  int64_t* digits;      // [18][M][N] or null
  int64_t* nonfinite;   // [M][N] or null
};

void gemm_rows(const GemmArgs& g, int64_t m0, int64_t m1) {
  for (int64_t m = m0; m < m1; ++m) {
    for (int64_t n = 0; n < g.N; ++n) {
      Big acc;
      big_zero(acc);
      int64_t nf = 0;
      for (int64_t k = 0; k < g.K; ++k) {
        double a = load_elem(g.dtype, g.A, m * g.sAm + k * g.sAk);
        double b = load_elem(g.dtype, g.B, n * g.sBn + k * g.sBk);
        if (!std::isfinite(a) || !std::isfinite(b)) {
          ++nf;
          continue;
        }
        add_exact_double(acc, a * b);
      }
      if (g.C) {
        float r;
        if (nf > 0) {
          uint32_t nan_bits = 0x7FC00000u;
          std::memcpy(&r, &nan_bits, sizeof(r));
        } else {
          r = big_round_to_f32(acc);
        }
        g.C[m * g.ldc + n] = r;
      }
      if (g.digits) big_to_digits(acc, g.digits + m * g.N + n, g.M * g.N);
      if (g.nonfinite) g.nonfinite[m * g.N + n] = nf;
    }
  }
}

template <class F>
void parallel_rows(int64_t rows, int nthreads, F&& body) {
  if (nthreads < 1) nthreads = 1;
  int64_t nt = std::min<int64_t>(nthreads, std::max<int64_t>(rows, 1));
  if (nt <= 1) {
    body(0, rows);
    return;
  }
  std::vector<std::thread> pool;
  int64_t chunk = (rows + nt - 1) / nt;
  for (int64_t t = 0; t < nt; ++t) {
    int64_t r0 = t * chunk, r1 = std::min(rows, r0 + chunk);
    if (r0 >= r1) break;
    pool.emplace_back([=, &body] { body(r0, r1); });
  }
  for (auto& th : pool) th.join();
}

// Sum arbitrary int64 digits (digit j weighs 2^(32j-298)) exactly.
Big digits_to_big(const int64_t* planes, int64_t idx, int64_t count) {
  Big acc;
  big_zero(acc);
  for (int j = 0; j < kDigits; ++j) {
    int64_t d = planes[j * count + idx];
    if (d > 0) big_add(acc, static_cast<uint64_t>(d), 32 * j);
    else if (d < 0) big_sub(acc, static_cast<uint64_t>(-(d + 1)) + 1u, 32 * j);
  }
  return acc;
}

}  // namespace

extern "C" {

int oracle_version() { return 1; }

// C[m,n] = RNE_f32( sum_k A(m,k) * B(n,k) ), A(m,k) = A[m*sAm + k*sAk],
// B(n,k) = B[n*sBn + k*sBk]; dtype 0 = f32, 1 = bf16 (raw 16-bit patterns).
// digits (optional): canonical [18][M][N]; nonfinite (optional): [M][N].
int oracle_gemm(int dtype, int64_t M, int64_t N, int64_t K, const void* A, int64_t sAm,
                int64_t sAk, const void* B, int64_t sBn, int64_t sBk, float* C, int64_t ldc,
                int64_t* digits, int64_t* nonfinite, int nthreads) {
  if (dtype != 0 && dtype != 1) return 1;
  if (M < 0 || N < 0 || K < 0) return 2;
  GemmArgs g{dtype, M, N, K, A, sAm, sAk, B, sBn, sBk, C, ldc, digits, nonfinite};
  parallel_rows(M, nthreads, [&](int64_t r0, int64_t r1) { gemm_rows(g, r0, r1); });
  return 0;
}

// Round digit arrays once: planes is [20][count] (18 digits, product count,
// non-finite count).  Any int64 digits are accepted; the value is their exact
// weighted sum.
int oracle_finalize(int64_t count, const int64_t* planes, float* out, int nthreads) {
  parallel_rows(count, nthreads, [&](int64_t r0, int64_t r1) {
    for (int64_t i = r0; i < r1; ++i) {
      if (planes[(kPlanes - 1) * count + i] != 0) {
        uint32_t nan_bits = 0x7FC00000u;
        std::memcpy(&out[i], &nan_bits, sizeof(float));
        continue;
      }
      out[i] = big_round_to_f32(digits_to_big(planes, i, count));
    }
  });
  return 0;
}

// Canonical form of arbitrary digit arrays; planes 18 and 19 are copied.
int oracle_canonicalize(int64_t count, const int64_t* planes, int64_t* out, int nthreads) {
  parallel_rows(count, nthreads, [&](int64_t r0, int64_t r1) {
    for (int64_t i = r0; i < r1; ++i) {
      big_to_digits(digits_to_big(planes, i, count), out + i, count);
      out[kDigits * count + i] = planes[kDigits * count + i];
      out[(kDigits + 1) * count + i] = planes[(kDigits + 1) * count + i];
    }
  });
  return 0;
}

}  // extern "C"
