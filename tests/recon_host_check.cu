// Host check of two reconstruction routines that are host-and-device code.
// 1. The CRT sum (crt_s128, det_crt.cuh): for each compiled count of moduli,
//    integers S with |S| below the bound the moduli count keeps
//    (M / (2 (1 + 2^-7)), M the product of the moduli) are reduced to
//    balanced residues and rebuilt; the result must equal S exactly.  Random
//    values of every magnitude plus the extremes.
// 2. The fast rounding of a 64-bit window (f32_bits_of_top, det_arith.cuh):
//    the binary32 pattern of t in [2^63, 2^64) must equal the host's own
//    round-to-nearest-even conversion, on random windows and on every tie.
// Prints "mismatches <n>" and exits nonzero on any mismatch.  Built with nvcc
// as host code only.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <random>

#include "det_arith.cuh"
#include "det_crt.cuh"

namespace {

typedef __int128 i128;
typedef unsigned __int128 u128;

i128 product(int P) {
  i128 m = 1;
  for (int i = 0; i < P; ++i) m *= det::modulus(i);
  return m;
}

template <int P>
long check(std::mt19937_64& g, long n) {
  const i128 M = product(P);
  const i128 bound = M * 64 / 129;                   // floor(M / (2 (1 + 2^-7)))
  long bad = 0;
  for (long t = 0; t < n; ++t) {
    i128 S;
    switch (t % 6) {
      case 0: S = bound; break;
      case 1: S = -bound; break;
      case 2: S = static_cast<i128>(g() % 5) - 2; break;
      default: {
        const u128 u = (static_cast<u128>(g()) << 64) | g();
        S = static_cast<i128>(u % static_cast<u128>(2 * bound + 1)) - bound;
        if (t % 6 == 3) S >>= static_cast<int>(g() % 96);   // every magnitude
      }
    }
    int32_t r[det::kNumModuli] = {};
    for (int i = 0; i < P; ++i) {
      const int p = det::modulus(i);
      long long v = static_cast<long long>(S % p);
      if (v < 0) v += p;
      if (v > (p - 1) / 2) v -= p;
      r[i] = static_cast<int32_t>(v);
    }
    uint64_t lo, hi;
    det::crt_s128<P>(r, lo, hi);
    const i128 got = static_cast<i128>((static_cast<u128>(hi) << 64) | lo);
    if (got != S) ++bad;
  }
  return bad;
}

long check_rounding(std::mt19937_64& g, long n) {
  long bad = 0;
  for (long t = 0; t < n; ++t) {
    uint64_t w = g() | (uint64_t(1) << 63);              // a window in [2^63, 2^64)
    switch (t % 4) {
      case 0: w = (w & ~((uint64_t(1) << 40) - 1)) | (uint64_t(1) << 39); break;   // a tie
      case 1: w |= (uint64_t(1) << 40) - 1; break;      // just below the next value
      default: break;
    }
    const float f = static_cast<float>(w);              // the host rounds to nearest even
    uint32_t want;
    std::memcpy(&want, &f, sizeof(want));
    if (det::f32_bits_of_top(w) != want) ++bad;
  }
  // the largest windows round up to 2^64
  const float top = static_cast<float>(~uint64_t(0));
  uint32_t want_top;
  std::memcpy(&want_top, &top, sizeof(want_top));
  if (det::f32_bits_of_top(~uint64_t(0)) != want_top) ++bad;
  return bad;
}

}  // namespace

int main() {
  std::mt19937_64 g(20261202);
  const long n = 300000;
  long bad = 0;
  bad += check<8>(g, n);
  bad += check<9>(g, n);
  bad += check<10>(g, n);
  bad += check<12>(g, n);
  bad += check<13>(g, n);
  bad += check<14>(g, n);
  bad += check_rounding(g, 4 * n);
  std::printf("mismatches %ld\n", bad);
  return bad != 0;
}
