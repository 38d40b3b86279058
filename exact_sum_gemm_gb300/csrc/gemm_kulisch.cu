// General exact GEMM kernel: every output owns a full Kulisch accumulator of
// 18 int64 digits (radix 2^32) in shared memory.
//
// det-train page, section "Method": each product is formed exactly and its
// base-2^32 limbs are integer-added into the output's digits.  Here a product
// p = mA * mB * 2^(eA+eB) (|mA*mB| < 2^48) is placed at bit offset
// off = eA + eB + 298 of the accumulator: digit j = off / 32 receives the low
// 32 bits of (mA*mB) << (off % 32) and digit j+1 the (signed) rest.  Digits
// are int64 with deferred carries; a product adds less than 2^47 to a digit,
// so the digits are carry-normalised every 2^15 products, well before any
// could leave int64.
//
// This kernel is exact for any exponent spread; its cost per product is two
// shared-memory read-modify-writes.  Tile: 32x32 outputs per 256-thread CTA,
// each thread owning 2x2 outputs and their 18 digits (147 KB of shared
// memory per CTA); K is staged in chunks of 32, decoded once per chunk into
// (signed significand, exponent) pairs, double-buffered.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "det_arith.cuh"
#include "det_gemm_internal.cuh"
#include "det_kernels.h"

namespace det {
namespace {

constexpr int kBM = 32;
constexpr int kBN = 32;
constexpr int kBK = 32;
constexpr int kThreads = 256;
constexpr int kOutputs = kBM * kBN;                 // 1024 outputs per CTA
constexpr int kPad = kBM + 1;                       // staging row stride (bank spread)
constexpr int kNormChunks = (1 << 15) / kBK;        // normalise every 2^15 products
constexpr int kMaxSplits = 64;                      // K-splits of one tile (their sum < 2^39)

constexpr size_t kAccBytes = size_t(kDigits) * kOutputs * sizeof(int64_t);
constexpr size_t kStageBytes = size_t(2) * kBK * kPad * sizeof(int2);
constexpr size_t kFlagBytes = size_t(2) * kBK * kBM;
constexpr size_t kSmemBytes = kAccBytes + 2 * kStageBytes + 2 * kFlagBytes;

struct alignas(16) Staging {
  uint32_t a[4];
  uint32_t b[4];
};

// One exact product into one output's digits (acc_o points at digit 0;
// digit j lives at acc_o[j * kOutputs]).
__device__ __forceinline__ void mac_digits(int64_t* acc_o, int2 a, int2 b) {
  const int off = a.y + b.y;                                  // bit offset of the product's LSB
  const int64_t prod = static_cast<int64_t>(a.x) * static_cast<int64_t>(b.x);
  const uint32_t p0 = static_cast<uint32_t>(prod);
  const uint32_t p1 = static_cast<uint32_t>(static_cast<uint64_t>(prod) >> 32);
  const uint32_t sx = static_cast<uint32_t>(static_cast<int32_t>(p1) >> 31);
  const uint32_t lo = __funnelshift_l(0u, p0, off);           // bits [0,32) of prod << r
  const uint32_t h0 = __funnelshift_l(p0, p1, off);           // bits [32,64)
  const uint32_t h1 = __funnelshift_l(p1, sx, off);           // bits [64,96), sign-extended
  const int64_t hi = static_cast<int64_t>((static_cast<uint64_t>(h1) << 32) | h0);
  int64_t* d = acc_o + ((off >> 5) * kOutputs);
  d[0] += static_cast<int64_t>(lo);
  d[kOutputs] += hi;
}

__device__ __forceinline__ void normalise_in_place(int64_t* acc_o) {
  int64_t carry = 0;
#pragma unroll
  for (int j = 0; j < kDigits - 1; ++j) {
    int64_t v = acc_o[j * kOutputs] + carry;
    acc_o[j * kOutputs] = static_cast<int64_t>(static_cast<uint32_t>(v));
    carry = v >> 32;
  }
  acc_o[(kDigits - 1) * kOutputs] += carry;
}

// Persistent: each CTA loops over the 32x32 quarters of the 64x64 tiles
// listed in general (general[0] = their count), so a call with no such tile
// costs one launch.
template <int kBf16>
__global__ void __launch_bounds__(kThreads, 1) kulisch_smem_kernel(GemmArgs p, const int* general,
                                                                    int splits, int64_t* accg,
                                                                    unsigned* qdone) {
  extern __shared__ __align__(16) unsigned char smem[];
  int64_t* acc = reinterpret_cast<int64_t*>(smem);
  int2* As = reinterpret_cast<int2*>(smem + kAccBytes);
  int2* Bs = reinterpret_cast<int2*>(smem + kAccBytes + kStageBytes);
  uint8_t* nfA = smem + kAccBytes + 2 * kStageBytes;
  uint8_t* nfB = nfA + kFlagBytes;

  const int64_t parents_n = (p.N + 2 * kBN - 1) / (2 * kBN);
  const int64_t quarters = int64_t(*general) * 4;
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  __shared__ int last_split;
  // work items: (quarter, K-split); with splits > 1 each item adds its
  // normalised digits to the quarter's slot in accg with 64-bit atomics (an
  // exact integer sum, so the order does not matter) and the item that
  // completes the quarter rounds it
  const int64_t nchunks_all = (p.K + kBK - 1) / kBK;
  const int64_t chunks_per_split = (nchunks_all + splits - 1) / splits;

  for (int64_t item = blockIdx.x; item < quarters * splits; item += gridDim.x) {
  const int64_t w = item / splits;
  const int64_t split = item - w * splits;
  const int64_t parent = general[1 + (w >> 2)];
  const int64_t ptm = parent / parents_n;
  const int64_t tm = 2 * ptm + ((w >> 1) & 1);
  const int64_t tn = 2 * (parent - ptm * parents_n) + (w & 1);
  const int64_t m0 = tm * kBM, n0 = tn * kBN;
  if (m0 >= p.M || n0 >= p.N) continue;               // ragged edge: quarter outside
  const int64_t c_begin = split * chunks_per_split;
  const int64_t c_end = c_begin + chunks_per_split < nchunks_all ? c_begin + chunks_per_split
                                                                  : nchunks_all;

  __syncthreads();                                    // previous tile done with smem
  for (int i = tid; i < kDigits * kOutputs; i += kThreads) acc[i] = 0;

  // global -> registers (raw bits) for one K chunk
  auto load_chunk = [&](int64_t k0, Staging& st) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = tid + kThreads * u;
      // A
      {
        const int r = p.opA ? (idx & 31) : (idx >> 5);
        const int k = p.opA ? (idx >> 5) : (idx & 31);
        const int64_t gm = m0 + r, gk = k0 + k;
        st.a[u] = (gm < p.M && gk < p.K) ? load_bits<kBf16>(p.A, a_offset(p, gm, gk)) : 0u;
      }
      // B
      {
        const int r = p.opB ? (idx & 31) : (idx >> 5);
        const int k = p.opB ? (idx >> 5) : (idx & 31);
        const int64_t gn = n0 + r, gk = k0 + k;
        // (a strided batch: B's rows of the tile's entry)
        st.b[u] = (gn < p.N && gk < p.K) ? load_bits<kBf16>(p.B, b_offset(p, brow_of(p, m0, gn), gk))
                                         : 0u;
      }
    }
  };
  // registers -> decoded shared staging; returns whether any element is non-finite
  auto store_chunk = [&](int buf, const Staging& st) -> int {
    int any_nf = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = tid + kThreads * u;
      {
        const int r = p.opA ? (idx & 31) : (idx >> 5);
        const int k = p.opA ? (idx >> 5) : (idx & 31);
        const Decoded d = decode_f32_bits(st.a[u]);
        As[(buf * kBK + k) * kPad + r] = make_int2(d.m, d.e + kLsbBias);
        nfA[(buf * kBK + k) * kBM + r] = d.nonfinite;
        any_nf |= d.nonfinite;
      }
      {
        const int r = p.opB ? (idx & 31) : (idx >> 5);
        const int k = p.opB ? (idx >> 5) : (idx & 31);
        const Decoded d = decode_f32_bits(st.b[u]);
        Bs[(buf * kBK + k) * kPad + r] = make_int2(d.m, d.e);
        nfB[(buf * kBK + k) * kBN + r] = d.nonfinite;
        any_nf |= d.nonfinite;
      }
    }
    return any_nf;
  };

  int64_t* acc_o[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) acc_o[s] = acc + s * kThreads + tid;
  int nf_count[4] = {0, 0, 0, 0};

  const int64_t nchunks = c_end > c_begin ? c_end - c_begin : 0;
  Staging st;
  int cur_nf = 0;
  if (nchunks > 0) {
    load_chunk(c_begin * kBK, st);
    cur_nf = store_chunk(0, st);
  }
  cur_nf = __syncthreads_or(cur_nf);

  for (int64_t c = 0; c < nchunks; ++c) {
    const int buf = static_cast<int>(c & 1);
    if (c + 1 < nchunks) load_chunk((c_begin + c + 1) * kBK, st);

    const int2* Ab = As + buf * kBK * kPad;
    const int2* Bb = Bs + buf * kBK * kPad;
#pragma unroll 4
    for (int kk = 0; kk < kBK; ++kk) {
      const int2 a0 = Ab[kk * kPad + ty];
      const int2 a1 = Ab[kk * kPad + ty + 16];
      const int2 b0 = Bb[kk * kPad + tx];
      const int2 b1 = Bb[kk * kPad + tx + 16];
      mac_digits(acc_o[0], a0, b0);
      mac_digits(acc_o[1], a0, b1);
      mac_digits(acc_o[2], a1, b0);
      mac_digits(acc_o[3], a1, b1);
    }
    if (cur_nf) {
      const uint8_t* fa = nfA + buf * kBK * kBM;
      const uint8_t* fb = nfB + buf * kBK * kBN;
      for (int kk = 0; kk < kBK; ++kk) {
        const int a0 = fa[kk * kBM + ty], a1 = fa[kk * kBM + ty + 16];
        const int b0 = fb[kk * kBN + tx], b1 = fb[kk * kBN + tx + 16];
        nf_count[0] += a0 | b0;
        nf_count[1] += a0 | b1;
        nf_count[2] += a1 | b0;
        nf_count[3] += a1 | b1;
      }
    }
    if ((c + 1) % kNormChunks == 0) {
#pragma unroll
      for (int s = 0; s < 4; ++s) normalise_in_place(acc_o[s]);
    }
    int next_nf = 0;
    if (c + 1 < nchunks) next_nf = store_chunk(buf ^ 1, st);
    cur_nf = __syncthreads_or(next_nf);
  }

  if (splits > 1) {
    // this split's digits, normalised (words below 2^32, a small top digit),
    // into the quarter's slot; a sum of up to 64 stays far inside int64
    int64_t* slot = accg + w * (int64_t(kDigits + 1) * kOutputs);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      normalise_in_place(acc_o[s]);
      const int o = s * kThreads + tid;
#pragma unroll
      for (int j = 0; j < kDigits; ++j)
        atomicAdd(reinterpret_cast<unsigned long long*>(slot + j * kOutputs + o),
                  static_cast<unsigned long long>(acc_o[s][j * kOutputs]));
      if (nf_count[s])
        atomicAdd(reinterpret_cast<unsigned long long*>(slot + kDigits * kOutputs + o),
                  static_cast<unsigned long long>(nf_count[s]));
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) last_split = atomicAdd(qdone + w, 1u) == unsigned(splits - 1);
    __syncthreads();
    if (!last_split) continue;
    __threadfence();
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int o = s * kThreads + tid;
#pragma unroll
      for (int j = 0; j < kDigits; ++j) acc_o[s][j * kOutputs] = __ldcg(slot + j * kOutputs + o);
      nf_count[s] = static_cast<int>(__ldcg(slot + kDigits * kOutputs + o));
    }
  }

  // epilogue: normalise, then round once (det_gemm) or write the digits
  const int64_t MN = p.M * p.N;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int64_t m = m0 + ty + 16 * (s >> 1);
    const int64_t n = n0 + tx + 16 * (s & 1);
    if (m >= p.M || n >= p.N) continue;
    int64_t d[kDigits];
#pragma unroll
    for (int j = 0; j < kDigits; ++j) d[j] = acc_o[s][j * kOutputs];
    uint32_t w[kDigits - 1];
    int64_t top;
    normalise_digits(d, w, top);
    if (p.P) {
      int64_t* out = p.P + m * p.N + n;
#pragma unroll
      for (int j = 0; j < kDigits - 1; ++j) out[j * MN] = static_cast<int64_t>(w[j]);
      out[(kDigits - 1) * MN] = top;
      out[kDigits * MN] = p.K;
      out[(kDigits + 1) * MN] = nf_count[s];
    } else {
      const uint32_t bits = nf_count[s] ? kNanBits : round_to_f32_bits(w, top);
      reinterpret_cast<uint32_t*>(p.C)[c_row_offset(p, m) + n] = bits;
    }
  }
  }  // tile loop
}

template <int kBf16>
cudaError_t launch_kulisch_t(const GemmArgs& a, const int* general, bool allow_split,
                             cudaStream_t stream) {
  static PerDeviceOnce configured;                 // the attribute is per device
  cudaError_t ce = configured.run([](int) {
    return cudaFuncSetAttribute(kulisch_smem_kernel<kBf16>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kSmemBytes));
  });
  if (ce != cudaSuccess) return ce;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  const int64_t tiles = ((a.M + kBM - 1) / kBM) * ((a.N + kBN - 1) / kBN);
  // Too few 32x32 tiles to fill the GPU twice and a long K: split K among
  // CTAs (the routed tiles are at most all of them; their count is known on
  // the device only).  The splits' digits meet in a zeroed pool slot per
  // quarter of every 64x64 tile.
  // The count is the one that fills the grid's waves best, at least 1024 of
  // K per split (each item zeroes its accumulator and adds it atomically).
  int splits = 1;
  if (allow_split && tiles < 2 * int64_t(sms) && a.K >= 2 * 1024) {
    const int64_t most = std::min<int64_t>(kMaxSplits, a.K / 1024);
    double best = 0.0;
    for (int64_t sp = 2; sp <= most; ++sp) {
      const int64_t items = tiles * sp;
      const int64_t waves = (items + sms - 1) / sms;
      const double fill = static_cast<double>(items) / static_cast<double>(waves * sms);
      if (fill > best + 1e-9) {
        best = fill;
        splits = static_cast<int>(sp);
      }
    }
  }
  int64_t* accg = nullptr;
  unsigned* qdone = nullptr;
  void* scratch = nullptr;
  if (splits > 1) {
    const int64_t slots = 4 * ((a.M + 2 * kBM - 1) / (2 * kBM)) * ((a.N + 2 * kBN - 1) / (2 * kBN));
    const size_t acc_bytes = sizeof(int64_t) * size_t(slots) * (kDigits + 1) * kOutputs;
    const size_t bytes = acc_bytes + sizeof(unsigned) * size_t(slots);
    cudaError_t e = pool_alloc(&scratch, bytes, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(scratch, 0, bytes, stream);
    if (e != cudaSuccess) {
      cudaFreeAsync(scratch, stream);
      return e;
    }
    accg = static_cast<int64_t*>(scratch);
    qdone = reinterpret_cast<unsigned*>(static_cast<char*>(scratch) + acc_bytes);
  }
  const int64_t items = tiles * splits;
  const int64_t grid = items < sms ? items : sms;
  kulisch_smem_kernel<kBf16><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(
      a, general, splits, accg, qdone);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (scratch != nullptr) {
    const cudaError_t f = cudaFreeAsync(scratch, stream);
    if (e == cudaSuccess) e = f;
  }
  return e;
}

}  // namespace

cudaError_t launch_kulisch(const GemmArgs& a, const int* general, bool allow_split,
                           cudaStream_t stream) {
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  return a.bf16 ? launch_kulisch_t<1>(a, general, allow_split, stream)
                : launch_kulisch_t<0>(a, general, allow_split, stream);
}

}  // namespace det
