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

constexpr int kThreads = 256;
constexpr int kTileRows = 32;
constexpr int kTileK = 64;

// Balanced residue of the signed integer m * 2^s (|m| < 2^24, 0 <= s <= 15)
// modulo the compile-time modulus p: a value in [-(p-1)/2, (p-1)/2].
template <int p>
__device__ __forceinline__ int balanced_residue(int32_t m, int s) {
  const uint32_t am = static_cast<uint32_t>(m < 0 ? -m : m);
  const uint32_t r = ((am % p) * ((1u << s) % p)) % p;
  int v = static_cast<int>(r);
  if (m < 0) v = -v;
  if (v > (p - 1) / 2) v -= p;
  if (v < -(p - 1) / 2) v += p;
  return v;
}

template <int i>
__device__ __forceinline__ void write_residues(__nv_bfloat16* planes, int64_t plane_stride,
                                               int64_t off, int nplanes, int32_t m, int s,
                                               bool live) {
  if constexpr (i < kNumModuli) {
    if (i < nplanes) {
      const int v = live ? balanced_residue<modulus(i)>(m, s) : 0;
      planes[i * plane_stride + off] = __float2bfloat16_rn(static_cast<float>(v));
      write_residues<i + 1>(planes, plane_stride, off, nplanes, m, s, live);
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
    write_residues<0>(o.planes, plane_stride, gr * o.Kp + gk, nplanes, m_int, live ? s : 0, live);
    if (deep && gk < o.K) {
      const int slot = atomicAdd(o.list_count + gr, 1);
      if (slot < o.cap) o.list[gr * o.cap + slot] = make_uint2(static_cast<uint32_t>(gk), tile[r][k]);
    }
  }
}

// ---------------------------------------------------------------- reconstruction

struct U128 {
  uint32_t w[4];
};

__device__ __forceinline__ void mul_add_small(U128& x, uint32_t mul, uint32_t add) {
  uint64_t carry = add;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint64_t t = static_cast<uint64_t>(x.w[i]) * mul + carry;
    x.w[i] = static_cast<uint32_t>(t);
    carry = t >> 32;
  }
}

// Garner: mixed-radix digits v_i in [0, p_i) of the unique S in [0, prod p)
// with S = r_i (mod p_i); then S = v_0 + p_0 (v_1 + p_1 (v_2 + ...)).
template <int i>
__device__ __forceinline__ void garner_digits(const int (&r)[kNumModuli], int (&v)[kNumModuli],
                                              int nplanes) {
  if constexpr (i < kNumModuli) {
    if (i < nplanes) {
      constexpr int p = modulus(i);
      constexpr int inv = garner_inverse(i);
      // t = (v_0 + p_0 (v_1 + ... + p_{i-2} v_{i-1})) mod p
      int t = 0;
#pragma unroll
      for (int j = i - 1; j >= 0; --j) t = (t * (modulus(j) % p) + v[j]) % p;
      int d = (r[i] - t) % p;
      if (d < 0) d += p;
      v[i] = (d * inv) % p;
      garner_digits<i + 1>(r, v, nplanes);
    }
  }
}

__device__ __forceinline__ void add_shifted_u128(int64_t (&d)[kDigits], U128 x, bool neg, int off) {
  // d += (neg ? -x : x) * 2^off, with 0 <= off; x < 2^103
  if (neg) {  // two's complement of the 128-bit magnitude
    uint32_t c = 1;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = ~x.w[i] + c;
      c = (c && v == 0u) ? 1u : 0u;
      x.w[i] = v;
    }
  }
  const uint32_t sx = neg ? 0xFFFFFFFFu : 0u;
  const int j = off >> 5, sh = off & 31;
  int64_t y[5];
  y[0] = static_cast<int64_t>(x.w[0] << sh);
  y[1] = static_cast<int64_t>(__funnelshift_l(x.w[0], x.w[1], sh));
  y[2] = static_cast<int64_t>(__funnelshift_l(x.w[1], x.w[2], sh));
  y[3] = static_cast<int64_t>(__funnelshift_l(x.w[2], x.w[3], sh));
  y[4] = static_cast<int64_t>(static_cast<int32_t>(__funnelshift_l(x.w[3], sx, sh)));
#pragma unroll
  for (int pl = 0; pl < kDigits; ++pl) {
    const int u = pl - j;
    d[pl] += u == 0 ? y[0] : u == 1 ? y[1] : u == 2 ? y[2] : u == 3 ? y[3] : u == 4 ? y[4] : 0;
  }
  // a piece that would land on digit 18 is at most the sign extension of the
  // value (which fits in 576 bits): fold it into digit 17
  if (j + 4 == kDigits) d[kDigits - 1] += y[4] * (int64_t(1) << 32);
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

template <int kBf16>
__global__ void __launch_bounds__(kThreads) reconstruct_kernel(GemmArgs g, ReconArgs ra) {
  const int64_t MN = g.M * g.N;
  const int64_t tiles_n = (g.N + kTile - 1) / kTile;
  // product of the moduli in use, and half of it (balanced range)
  U128 mod_prod = {{1u, 0u, 0u, 0u}};
#pragma unroll
  for (int i = 0; i < kNumModuli; ++i)
    if (i < ra.nplanes) mul_add_small(mod_prod, modulus(i), 0u);
  U128 half = mod_prod;
#pragma unroll
  for (int i = 0; i < 3; ++i) half.w[i] = (half.w[i] >> 1) | (half.w[i + 1] << 31);
  half.w[3] >>= 1;
  const bool failed = ra.error != nullptr && *ra.error != 0;

  for (int64_t idx = int64_t(blockIdx.x) * kThreads + threadIdx.x; idx < MN;
       idx += int64_t(gridDim.x) * kThreads) {
    const int64_t m = idx / g.N, n = idx - (idx / g.N) * g.N;
    if (ra.route[(m / kTile) * tiles_n + n / kTile]) continue;   // general kernel's output
    int r[kNumModuli];
#pragma unroll
    for (int i = 0; i < kNumModuli; ++i) r[i] = i < ra.nplanes ? ra.res[i * MN + idx] : 0;
    int v[kNumModuli];
    garner_digits<0>(r, v, ra.nplanes);
    U128 s = {{0u, 0u, 0u, 0u}};
#pragma unroll
    for (int i = kNumModuli - 1; i >= 0; --i)
      if (i < ra.nplanes) mul_add_small(s, modulus(i), static_cast<uint32_t>(v[i]));
    // balanced: S >= prod/2 means S - prod (negative)
    bool ge = false, decided = false;
#pragma unroll
    for (int i = 3; i >= 0; --i) {
      if (!decided && s.w[i] != half.w[i]) {
        ge = s.w[i] > half.w[i];
        decided = true;
      }
    }
    // (s == half is non-negative: the product of odd moduli is odd)
    if (ge) {  // magnitude = prod - s
      uint32_t borrow = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint64_t t = static_cast<uint64_t>(mod_prod.w[i]) - s.w[i] - borrow;
        s.w[i] = static_cast<uint32_t>(t);
        borrow = static_cast<uint32_t>(t >> 63);
      }
    }
    int emA = ra.emaxA[m], emB = ra.emaxB[n];
    emA = emA == kEmaxEmpty ? 0 : emA;
    emB = emB == kEmaxEmpty ? 0 : emB;
    int64_t d[kDigits];
#pragma unroll
    for (int pl = 0; pl < kDigits; ++pl) d[pl] = 0;
    // shallow part: S * 2^(emA + emB - 30), placed at bit offset emA + emB - 30 + 298
    // (bf16 planes hold significands without their 16 zero bits: another 2^32)
    int off = emA + emB - 2 * kDeepGap + kLsbBias + (kBf16 ? 32 : 0);
    if (off < 0) {            // S is then a multiple of 2^-off: shift exactly
      const int sh = -off;
#pragma unroll
      for (int i = 0; i < 3; ++i) s.w[i] = __funnelshift_r(s.w[i], s.w[i + 1], sh);
      s.w[3] >>= sh;
      off = 0;
    }
    add_shifted_u128(d, s, ge, off);
    // deep elements of row m of A, with every element of column n of B
    int64_t nf = 0;
    const int na = min(ra.countA[m], ra.cap);
    for (int q = 0; q < na; ++q) {
      const uint2 ent = ra.listA[m * ra.cap + q];
      const int64_t k = ent.x;
      const Decoded a = decode_f32_bits(ent.y);
      const Decoded b = decode_f32_bits(
          load_bits<kBf16>(g.B, g.opB ? k * g.ldb + n : n * g.ldb + k));
      if (a.nonfinite || b.nonfinite) ++nf;
      else add_product(d, a.m, a.e, b.m, b.e);
    }
    // deep elements of column n of B, with the shallow (or zero) elements of row m
    const int nb = min(ra.countB[n], ra.cap);
    for (int q = 0; q < nb; ++q) {
      const uint2 ent = ra.listB[n * ra.cap + q];
      const int64_t k = ent.x;
      const Decoded b = decode_f32_bits(ent.y);
      const Decoded a = decode_f32_bits(
          load_bits<kBf16>(g.A, g.opA ? k * g.lda + m : m * g.lda + k));
      const bool a_listed = a.nonfinite || (a.m != 0 && a.e - emA + kDeepGap < 0);
      if (a_listed) continue;                             // counted with row m's list
      if (b.nonfinite) ++nf;
      else add_product(d, a.m, a.e, b.m, b.e);
    }
    uint32_t w[kDigits - 1];
    int64_t top;
    normalise_digits(d, w, top);
    if (failed) nf = 1;
    if (g.P) {
      int64_t* out = g.P + idx;
#pragma unroll
      for (int pl = 0; pl < kDigits - 1; ++pl) out[pl * MN] = static_cast<int64_t>(w[pl]);
      out[(kDigits - 1) * MN] = top;
      out[kDigits * MN] = g.K;
      out[(kDigits + 1) * MN] = nf;
    } else {
      reinterpret_cast<uint32_t*>(g.C)[m * g.ldc + n] = nf ? kNanBits : round_to_f32_bits(w, top);
    }
  }
}

int grid_for(int64_t work) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  const int64_t want = (work + kThreads - 1) / kThreads;
  const int64_t cap = int64_t(sms) * 8;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
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

cudaError_t launch_reconstruct(const GemmArgs& g, const ReconArgs& ra, cudaStream_t stream) {
  const int64_t MN = g.M * g.N;
  if (MN == 0) return cudaSuccess;
  if (g.bf16) reconstruct_kernel<1><<<grid_for(MN), kThreads, 0, stream>>>(g, ra);
  else reconstruct_kernel<0><<<grid_for(MN), kThreads, 0, stream>>>(g, ra);
  note_launch();
  return cudaGetLastError();
}

}  // namespace det
