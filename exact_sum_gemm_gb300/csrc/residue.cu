// Residue (CRT) decomposition of the exact GEMM, the CUDA-core halves:
//   residue_kernel      operands -> bf16 residue planes + per-row deep lists
//   reconstruct_kernel  residues of the shallow dot product -> exact value
//                       (Garner CRT) + deep products -> digits -> round once
//
// Shallow elements.  For a row r of an operand with largest last-bit exponent
// emax[r], an element m*2^e with e >= emax[r] - 15 is the integer
//     X_int = m * 2^(e - emax[r] + 15),   |X_int| < 2^39 (f32), 2^23 (bf16,
//     whose significand has 8 bits), times 2^(emax[r] - 15).  So for an output (m, n) the shallow products sum to
//     2^(emaxA[m] + emaxB[n] - 30) * S,   S = sum_k A_int[m,k] * B_int[n,k],
// an exact integer dot product with |S| < K * 2^78.  S is computed modulo
// kNumModuli small odd pairwise-coprime moduli (residues in bf16 planes,
// multiplied on tensor cores with exact fp32 accumulation) and rebuilt here
// by the Chinese remainder theorem: the moduli's product exceeds 2|S|.
// Deep elements (more than 15 binades below the row max) and non-finite ones
// are left out of the planes and listed per row; their products are added
// exactly, one by one, during reconstruction.  Together this is exactly the
// det-train page's "exact fp64-product sum rounded once to fp32" (section
// "Method"); only the order of the exact integer additions differs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "det_arith.cuh"
#include "det_gemm_internal.cuh"
#include "det_kernels.h"
#include "det_residue.cuh"

namespace det {
namespace {

struct CrtTable {
  uint32_t c[kNumModuli][4];   // CRT weights C_i, 128-bit, least significant limb first
  uint32_t m[4];               // M = product of the moduli in use
  float frac[kNumModuli];      // C_i / M, to estimate the quotient of sum r_i C_i by M
};

constexpr int kThreads = 256;
constexpr int kTileRows = 32;
constexpr int kTileK = 64;

// x mod p for an integer-valued float 0 <= x < 2^24 (every step exact: the
// quotient estimate is off by at most one and the fma remainder is exact).
template <int p>
__device__ __forceinline__ float fmod_exact(float x) {
  constexpr float fp = static_cast<float>(p);
  constexpr float inv = 1.0f / static_cast<float>(p);
  const float q = floorf(x * inv);
  float r = fmaf(-q, fp, x);
  r = r < 0.0f ? r + fp : r;
  r = r >= fp ? r - fp : r;
  return r;
}

// Balanced residue of the signed integer m * 2^s (|m| < 2^24, 0 <= s <= 15)
// modulo the compile-time modulus p: a value in [-(p-1)/2, (p-1)/2].
template <int p>
__device__ __forceinline__ float balanced_residue(int32_t m, float pow2s) {
  const float am = static_cast<float>(m < 0 ? -m : m);              // exact
  const float r = fmod_exact<p>(fmod_exact<p>(am) * fmod_exact<p>(pow2s));   // < 2^16 before mod
  float v = m < 0 ? -r : r;
  constexpr float h = static_cast<float>((p - 1) / 2);
  v = v > h ? v - static_cast<float>(p) : v;
  v = v < -h ? v + static_cast<float>(p) : v;
  return v;
}

template <int i>
__device__ __forceinline__ void write_residues(__nv_bfloat16* planes, int64_t plane_stride,
                                               int64_t off, int nplanes, int32_t m, float pow2s,
                                               bool live) {
  if constexpr (i < kNumModuli) {
    if (i < nplanes) {
      const float v = live ? balanced_residue<modulus(i)>(m, pow2s) : 0.0f;
      planes[i * plane_stride + off] = __float2bfloat16_rn(v);        // |v| <= 127: exact
      write_residues<i + 1>(planes, plane_stride, off, nplanes, m, pow2s, live);
    }
  }
}

// One block: 32 rows x 64 k of one operand.  Planes are [P][rows][Kp].
template <int kBf16>
__global__ void __launch_bounds__(kThreads) residue_kernel(ResidueOperand o, int nplanes) {
  __shared__ uint32_t tile[kTileRows][kTileK + 1];
  const int tid = threadIdx.x;
  const int64_t r0 = int64_t(blockIdx.y) * kTileRows;
  const int64_t k0 = int64_t(blockIdx.x) * kTileK;
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
  __syncthreads();
  const int64_t plane_stride = o.rows * o.Kp;
#pragma unroll 1
  for (int u = 0; u < kTileRows * kTileK / kThreads; ++u) {
    const int idx = tid + u * kThreads;
    const int r = idx >> 6, k = idx & 63;
    const int64_t gr = r0 + r, gk = k0 + k;
    if (gr >= o.rows || gk >= o.Kp) continue;
    const Decoded d = decode_f32_bits(tile[r][k]);
    int em = o.emax[gr];
    em = em == kEmaxEmpty ? 0 : em;
    const int s = d.e - em + kDeepGap;
    const bool deep = d.nonfinite || (d.m != 0 && s < 0);
    const bool live = !deep && d.m != 0;
    // a bf16 significand widened to binary32 carries 16 zero bits: drop them
    // (exactly) so that |X_int| < 2^23; the reconstruction scales back by 2^32
    const int32_t m_int = kBf16 ? (d.m >> 16) : d.m;
    const float pow2s = __int_as_float((127 + (live ? s : 0)) << 23);   // 2^s, exact
    write_residues<0>(o.planes, plane_stride, gr * o.Kp + gk, nplanes, m_int, pow2s, live);
    if (deep && gk < o.K) {
      const int slot = atomicAdd(o.list_count + gr, 1);
      if (slot < o.cap) o.list[gr * o.cap + slot] = make_uint2(static_cast<uint32_t>(gk), tile[r][k]);
    }
  }
}

// ---------------------------------------------------------------- reconstruction
//
// Per output (m, n) on a residue-path tile:
//   S   = the unique integer with S = r_i (mod p_i), |S| < M/2 (M = prod p_i),
//         by the CRT sum  S' = sum_i r_i C_i,  C_i = (M/p_i) * ((M/p_i)^-1 mod p_i),
//         S = S' mod M (balanced);
//   T   = S * 2^64 plus every product involving a deep element, exact, as a
//         192-bit two's-complement integer whose bit 0 weighs 2^E with
//         E = emaxA + emaxB - 30 - 64 (+32 for bf16 planes);
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
    const int wi = p >> 6, r = p & 63;
    const uint64_t lo = wi == 0 ? t.w[0] : (wi == 1 ? t.w[1] : t.w[2]);
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

// Cold path of one output: the digit route.  Used for det_gemm_partial (the
// digits are the output) and when a deep product falls outside the 192-bit
// window; rebuilds the exact value as 18 int64 digits and writes it.
template <int kBf16>
__device__ __noinline__ void output_via_digits(const GemmArgs& g, const ReconArgs& ra, int64_t m,
                                               int64_t n, W192 t, int E, bool wide, __int128 S,
                                               int emA, int64_t nf) {
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
    const int nb = min(ra.countB[n], ra.cap);
    for (int q = 0; q < na; ++q) {
      const uint2 ent = ra.listA[m * ra.cap + q];
      const int64_t k = ent.x;
      const Decoded a = decode_f32_bits(ent.y);
      const Decoded b = decode_f32_bits(load_bits<kBf16>(g.B, g.opB ? k * g.ldb + n : n * g.ldb + k));
      if (!a.nonfinite && !b.nonfinite) add_product(d, a.m, a.e, b.m, b.e);
    }
    for (int q = 0; q < nb; ++q) {
      const uint2 ent = ra.listB[n * ra.cap + q];
      const int64_t k = ent.x;
      const Decoded b = decode_f32_bits(ent.y);
      const Decoded a = decode_f32_bits(load_bits<kBf16>(g.A, g.opA ? k * g.lda + m : m * g.lda + k));
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
    reinterpret_cast<uint32_t*>(g.C)[m * g.ldc + n] = nf ? kNanBits : round_to_f32_bits(w, top);
  }
}

// S = the balanced CRT value of residues r (one per modulus in use).
__device__ __forceinline__ __int128 crt_balanced(const uint32_t (&r)[kNumModuli], int P,
                                                 const CrtTable& crt) {
  uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  float qf = 0.0f;
#pragma unroll
  for (int i = 0; i < kNumModuli; ++i) {
    if (i < P) {
      // (a3:a2:a1:a0) += r_i * C_i   (r_i < 256, C_i < M < 2^103; sum < 2^115)
      uint64_t t = static_cast<uint64_t>(crt.c[i][0]) * r[i] + a0;
      a0 = static_cast<uint32_t>(t);
      t = static_cast<uint64_t>(crt.c[i][1]) * r[i] + a1 + (t >> 32);
      a1 = static_cast<uint32_t>(t);
      t = static_cast<uint64_t>(crt.c[i][2]) * r[i] + a2 + (t >> 32);
      a2 = static_cast<uint32_t>(t);
      a3 = crt.c[i][3] * r[i] + a3 + static_cast<uint32_t>(t >> 32);
      qf = fmaf(static_cast<float>(r[i]), crt.frac[i], qf);     // ~ acc / M
    }
  }
  // quotient estimate within one of floor(acc / M); remainder by one multiply
  const uint32_t q = static_cast<uint32_t>(qf);
  uint64_t t = static_cast<uint64_t>(crt.m[0]) * q;
  const uint32_t p0 = static_cast<uint32_t>(t);
  t = static_cast<uint64_t>(crt.m[1]) * q + (t >> 32);
  const uint32_t p1 = static_cast<uint32_t>(t);
  t = static_cast<uint64_t>(crt.m[2]) * q + (t >> 32);
  const uint32_t p2 = static_cast<uint32_t>(t);
  const uint32_t p3 = crt.m[3] * q + static_cast<uint32_t>(t >> 32);
  const u128 acc = (static_cast<u128>(a3) << 96) | (static_cast<u128>(a2) << 64) |
                   (static_cast<u128>(a1) << 32) | a0;
  const u128 qm = (static_cast<u128>(p3) << 96) | (static_cast<u128>(p2) << 64) |
                  (static_cast<u128>(p1) << 32) | p0;
  const u128 M = (static_cast<u128>(crt.m[3]) << 96) | (static_cast<u128>(crt.m[2]) << 64) |
                 (static_cast<u128>(crt.m[1]) << 32) | crt.m[0];
  __int128 rem = static_cast<__int128>(acc - qm);
  if (rem < 0) rem += static_cast<__int128>(M);
  else if (rem >= static_cast<__int128>(M)) rem -= static_cast<__int128>(M);
  return rem > static_cast<__int128>(M >> 1) ? rem - static_cast<__int128>(M) : rem;
}

constexpr int kReconCols = 4;                       // outputs per thread (one row)

template <int kBf16>
__global__ void __launch_bounds__(kThreads, 2) reconstruct_kernel(GemmArgs g, ReconArgs ra,
                                                                const __grid_constant__ CrtTable crt) {
  const int64_t MN = g.M * g.N;
  const int64_t tiles_n = (g.N + kTile - 1) / kTile;
  const bool failed = ra.error != nullptr && *ra.error != 0;
  const int64_t n0 = (int64_t(blockIdx.x) * kThreads + threadIdx.x) * kReconCols;
  if (n0 >= g.N) return;
  const int ncols = g.N - n0 < kReconCols ? static_cast<int>(g.N - n0) : kReconCols;

  for (int64_t m = blockIdx.y; m < g.M; m += gridDim.y) {
    if (ra.route[(m / kTile) * tiles_n + n0 / kTile]) continue;   // general kernel's outputs
    int emA = ra.emaxA[m];
    emA = emA == kEmaxEmpty ? 0 : emA;
    const int na = min(ra.countA[m], ra.cap);
    const int64_t base = m * g.N + n0;
    // residues of the (up to) four outputs: one packed word per plane
    uint32_t packed[kNumModuli];
    // word loads need every plane's address 4-byte aligned: base and M*N both
    // multiples of 4 (the residue buffer itself is 1024-byte aligned)
    const bool vec = ncols == kReconCols && ((base | MN) & 3) == 0 &&
                     (reinterpret_cast<uintptr_t>(ra.res) & 3u) == 0;
#pragma unroll
    for (int i = 0; i < kNumModuli; ++i) {
      packed[i] = 0;
      if (i < ra.nplanes) {
        const uint8_t* plane = ra.res + i * MN + base;
        if (vec) {
          packed[i] = *reinterpret_cast<const uint32_t*>(plane);
        } else {
#pragma unroll
          for (int j = 0; j < kReconCols; ++j)
            if (j < ncols) packed[i] |= static_cast<uint32_t>(plane[j]) << (8 * j);
        }
      }
    }
#pragma unroll 1
    for (int j = 0; j < ncols; ++j) {
      const int64_t n = n0 + j;
      uint32_t rj[kNumModuli];                      // this output's residues
#pragma unroll
      for (int i = 0; i < kNumModuli; ++i) rj[i] = (packed[i] >> (8 * j)) & 0xFFu;
      const __int128 S = crt_balanced(rj, ra.nplanes, crt);
      int emB = ra.emaxB[n];
      emB = emB == kEmaxEmpty ? 0 : emB;
      const int E = emA + emB - 2 * kDeepGap + (kBf16 ? 32 : 0) - 64;
      W192 t;
      t.w[0] = 0;
      t.w[1] = static_cast<uint64_t>(S);
      t.w[2] = static_cast<uint64_t>(S >> 64);
      int64_t nf = 0;
      bool wide = false;
      const int nb = min(ra.countB[n], ra.cap);
      // deep elements: row m of A with every element of column n of B, then
      // column n of B with the shallow (or zero) elements of row m
      for (int q = 0; q < na; ++q) {
        const uint2 ent = ra.listA[m * ra.cap + q];
        const int64_t k = ent.x;
        const Decoded a = decode_f32_bits(ent.y);
        const Decoded b =
            decode_f32_bits(load_bits<kBf16>(g.B, g.opB ? k * g.ldb + n : n * g.ldb + k));
        if (a.nonfinite || b.nonfinite) {
          ++nf;
        } else if (a.m != 0 && b.m != 0) {
          const int sh = a.e + b.e - E;
          if (sh < 0 || sh > 140) wide = true;
          else w192_add_shifted(t, static_cast<int64_t>(a.m) * b.m, sh);
        }
      }
      for (int q = 0; q < nb; ++q) {
        const uint2 ent = ra.listB[n * ra.cap + q];
        const int64_t k = ent.x;
        const Decoded b = decode_f32_bits(ent.y);
        const Decoded a =
            decode_f32_bits(load_bits<kBf16>(g.A, g.opA ? k * g.lda + m : m * g.lda + k));
        if (a.nonfinite || (a.m != 0 && a.e - emA + kDeepGap < 0)) continue;  // row m's list had it
        if (b.nonfinite) {
          ++nf;
        } else if (a.m != 0 && b.m != 0) {
          const int sh = a.e + b.e - E;
          if (sh < 0 || sh > 140) wide = true;
          else w192_add_shifted(t, static_cast<int64_t>(a.m) * b.m, sh);
        }
      }
      if (failed) nf = 1;
      if (!wide && g.P == nullptr) {
        reinterpret_cast<uint32_t*>(g.C)[m * g.ldc + n] = nf ? kNanBits : round_w192(t, E);
      } else {
        output_via_digits<kBf16>(g, ra, m, n, t, E, wide, S, emA, nf);
      }
    }
  }
}


}  // namespace

int residue_planes_needed(const GemmArgs& g) {
  // |S| <= K * maxA * maxB with max = (2^bits - 1) * 2^15; need prod > 2|S|
  const unsigned __int128 sig = g.bf16 ? 0xFFu : 0xFFFFFFu;
  const unsigned __int128 mx = sig << kDeepGap;
  const unsigned __int128 bound = static_cast<unsigned __int128>(g.K > 0 ? g.K : 1) * mx * mx * 2;
  unsigned __int128 prod = 1;
  for (int i = 0; i < kNumModuli; ++i) {
    prod *= static_cast<unsigned>(modulus(i));
    if (prod > bound) return i + 1;
  }
  return -1;
}

cudaError_t launch_residues(const ResidueOperand& o, int bf16, int nplanes, cudaStream_t stream) {
  if (o.rows == 0 || o.Kp == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>((o.Kp + kTileK - 1) / kTileK),
            static_cast<unsigned>((o.rows + kTileRows - 1) / kTileRows));
  if (bf16) residue_kernel<1><<<grid, kThreads, 0, stream>>>(o, nplanes);
  else residue_kernel<0><<<grid, kThreads, 0, stream>>>(o, nplanes);
  note_launch();
  return cudaGetLastError();
}

CrtTable make_crt_table(int nplanes) {
  // M = prod p_i; C_i = (M/p_i) * ((M/p_i)^-1 mod p_i) mod M  (exact 128-bit host arithmetic)
  CrtTable t{};
  unsigned __int128 M = 1;
  for (int i = 0; i < nplanes; ++i) M *= static_cast<unsigned>(modulus(i));
  for (int i = 0; i < nplanes; ++i) {
    const unsigned p = static_cast<unsigned>(modulus(i));
    const unsigned __int128 Mi = M / p;
    const unsigned mi = static_cast<unsigned>(Mi % p);
    unsigned inv = 1;
    for (unsigned c = 1; c < p; ++c)
      if ((mi * c) % p == 1) {
        inv = c;
        break;
      }
    const unsigned __int128 C = (Mi * inv) % M;
    for (int w = 0; w < 4; ++w) t.c[i][w] = static_cast<uint32_t>(C >> (32 * w));
    t.frac[i] = static_cast<float>(static_cast<long double>(C) / static_cast<long double>(M));
  }
  for (int w = 0; w < 4; ++w) t.m[w] = static_cast<uint32_t>(M >> (32 * w));
  return t;
}

cudaError_t launch_reconstruct(const GemmArgs& g, const ReconArgs& ra, cudaStream_t stream) {
  const int64_t MN = g.M * g.N;
  if (MN == 0) return cudaSuccess;
  const CrtTable crt = make_crt_table(ra.nplanes);
  const int64_t cols_per_block = int64_t(kThreads) * kReconCols;
  dim3 grid(static_cast<unsigned>((g.N + cols_per_block - 1) / cols_per_block),
            static_cast<unsigned>(g.M < 65535 ? g.M : 65535));
  if (g.bf16) reconstruct_kernel<1><<<grid, kThreads, 0, stream>>>(g, ra, crt);
  else reconstruct_kernel<0><<<grid, kThreads, 0, stream>>>(g, ra, crt);
  note_launch();
  return cudaGetLastError();
}

}  // namespace det
