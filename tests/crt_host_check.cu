// Host check of the reconstruction's CRT sum (crt_s128, det_crt.cuh): for each
// compiled count of moduli, integers S with |S| below the bound the moduli
// count keeps (M / (2 (1 + 2^-7)), M the product of the moduli) are reduced
// to balanced residues and rebuilt; the result must equal S exactly.  Random
// values of every magnitude plus the extremes.  Prints "mismatches <n>" and
// exits nonzero on any mismatch.  Built with nvcc as host code only.
#include <cstdio>
#include <cstdint>
#include <random>

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
  std::printf("mismatches %ld\n", bad);
  return bad != 0;
}
