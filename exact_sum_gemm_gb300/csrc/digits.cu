// Digit-array kernels: combine (elementwise int64 addition of partials) and
// finalize (carry-normalise, round once to fp32).
//
// det-train page, section "Method": digit arrays of K-shards combine by plain
// addition, and the final digits get a single rounding to fp32 (to nearest,
// ties to even).  Both kernels are HBM-bound streams over planar [20][M][N] int64
// arrays: consecutive threads touch consecutive outputs of one plane, so every
// load and store is coalesced; where alignment allows, each thread handles two
// neighbouring outputs with 16-byte accesses.  Grids are a multiple of the SM
// count and loop over the outputs.
#include <cuda_runtime.h>
#include <stdint.h>

#include "det_arith.cuh"
#include "det_kernels.h"

namespace det {
namespace {

constexpr int kThreads = 256;

struct CombineArgs {
  const int64_t* parts[kMaxPartsPerLaunch];
  int n;
  int64_t count;        // outputs per plane (M*N)
  int64_t* out;
};

__device__ __forceinline__ void canonical_write(int64_t (&d)[kPlanes], int64_t* out, int64_t count,
                                                int64_t i) {
  int64_t carry = 0;
#pragma unroll
  for (int j = 0; j < kDigits - 1; ++j) {
    int64_t v = d[j] + carry;
    out[j * count + i] = static_cast<int64_t>(static_cast<uint32_t>(v));
    carry = v >> 32;
  }
  out[(kDigits - 1) * count + i] = d[kDigits - 1] + carry;
  out[kDigits * count + i] = d[kDigits];
  out[(kDigits + 1) * count + i] = d[kDigits + 1];
}

// Scalar variant: one output per thread per iteration.
__global__ void __launch_bounds__(kThreads) combine_kernel_1(CombineArgs a) {
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < a.count; i += stride) {
    int64_t d[kPlanes];
#pragma unroll
    for (int j = 0; j < kPlanes; ++j) d[j] = __ldg(a.parts[0] + j * a.count + i);
    for (int q = 1; q < a.n; ++q) {
#pragma unroll
      for (int j = 0; j < kPlanes; ++j) d[j] += __ldg(a.parts[q] + j * a.count + i);
    }
    canonical_write(d, a.out, a.count, i);
  }
}

// Vector variant: two neighbouring outputs per thread (count even, 16B-aligned planes).
__global__ void __launch_bounds__(kThreads) combine_kernel_2(CombineArgs a) {
  const int64_t pairs = a.count >> 1;
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < pairs; i += stride) {
    int64_t d0[kPlanes], d1[kPlanes];
#pragma unroll
    for (int j = 0; j < kPlanes; ++j) {
      const longlong2 v = __ldg(reinterpret_cast<const longlong2*>(a.parts[0] + j * a.count) + i);
      d0[j] = v.x;
      d1[j] = v.y;
    }
    for (int q = 1; q < a.n; ++q) {
#pragma unroll
      for (int j = 0; j < kPlanes; ++j) {
        const longlong2 v = __ldg(reinterpret_cast<const longlong2*>(a.parts[q] + j * a.count) + i);
        d0[j] += v.x;
        d1[j] += v.y;
      }
    }
    int64_t c0 = 0, c1 = 0;
#pragma unroll
    for (int j = 0; j < kDigits - 1; ++j) {
      const int64_t v0 = d0[j] + c0, v1 = d1[j] + c1;
      longlong2 o;
      o.x = static_cast<int64_t>(static_cast<uint32_t>(v0));
      o.y = static_cast<int64_t>(static_cast<uint32_t>(v1));
      c0 = v0 >> 32;
      c1 = v1 >> 32;
      reinterpret_cast<longlong2*>(a.out + j * a.count)[i] = o;
    }
    reinterpret_cast<longlong2*>(a.out + (kDigits - 1) * a.count)[i] =
        make_longlong2(d0[kDigits - 1] + c0, d1[kDigits - 1] + c1);
    reinterpret_cast<longlong2*>(a.out + kDigits * a.count)[i] =
        make_longlong2(d0[kDigits], d1[kDigits]);
    reinterpret_cast<longlong2*>(a.out + (kDigits + 1) * a.count)[i] =
        make_longlong2(d0[kDigits + 1], d1[kDigits + 1]);
  }
}

__device__ __forceinline__ uint32_t finalize_one(const int64_t (&d)[kDigits], int64_t nonfinite) {
  uint32_t w[kDigits - 1];
  int64_t top;
  normalise_digits(d, w, top);
  return nonfinite != 0 ? kNanBits : round_to_f32_bits(w, top);
}

__global__ void __launch_bounds__(kThreads) finalize_kernel_1(const int64_t* __restrict__ P,
                                                               int64_t M, int64_t N,
                                                               uint32_t* __restrict__ C,
                                                               int64_t ldc) {
  const int64_t count = M * N;
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < count; i += stride) {
    int64_t d[kDigits];
#pragma unroll
    for (int j = 0; j < kDigits; ++j) d[j] = __ldg(P + j * count + i);
    const int64_t nf = __ldg(P + (kDigits + 1) * count + i);
    const uint32_t bits = finalize_one(d, nf);
    if (ldc == N) {
      C[i] = bits;
    } else {
      const int64_t m = i / N;
      C[m * ldc + (i - m * N)] = bits;
    }
  }
}

// Four blocks per SM (64 registers; the compiler keeps a few words on the
// stack): the loads of more outputs in flight outweigh the spills (measured at
// 4096x4096: 0.474 -> 0.419 ms, 0.81 -> 0.92 of the copy peak).
__global__ void __launch_bounds__(kThreads, 4) finalize_kernel_2(const int64_t* __restrict__ P,
                                                               int64_t count,
                                                               uint2* __restrict__ C) {
  const int64_t pairs = count >> 1;
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < pairs; i += stride) {
    int64_t d0[kDigits], d1[kDigits];
#pragma unroll
    for (int j = 0; j < kDigits; ++j) {
      const longlong2 v = __ldg(reinterpret_cast<const longlong2*>(P + j * count) + i);
      d0[j] = v.x;
      d1[j] = v.y;
    }
    const longlong2 nf = __ldg(reinterpret_cast<const longlong2*>(P + (kDigits + 1) * count) + i);
    C[i] = make_uint2(finalize_one(d0, nf.x), finalize_one(d1, nf.y));
  }
}

int grid_for(int64_t work) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  const int64_t want = (work + kThreads - 1) / kThreads;
  const int64_t cap = int64_t(sms) * 8;             // 8 resident CTAs of 256 threads per SM
  int64_t g = want < cap ? want : cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_combine(const int64_t* const* parts, int n, int64_t count, int64_t* out,
                           cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  // The first launch sums up to 16 parts into out; each later launch folds
  // out itself plus up to 15 more parts (re-normalising every time).
  int done = 0;
  bool first = true;
  while (done < n) {
    CombineArgs a;
    int k = 0;
    if (!first) a.parts[k++] = out;
    while (k < kMaxPartsPerLaunch && done < n) a.parts[k++] = parts[done++];
    a.n = k;
    a.count = count;
    a.out = out;
    bool vec = (count % 2 == 0) && aligned16(out);
    for (int q = 0; q < k; ++q) vec = vec && aligned16(a.parts[q]);
    if (vec) {
      combine_kernel_2<<<grid_for(count / 2), kThreads, 0, stream>>>(a);
    } else {
      combine_kernel_1<<<grid_for(count), kThreads, 0, stream>>>(a);
    }
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    first = false;
  }
  return cudaSuccess;
}

cudaError_t launch_finalize(const int64_t* P, int64_t M, int64_t N, float* C, int64_t ldc,
                            cudaStream_t stream) {
  const int64_t count = M * N;
  if (count == 0) return cudaSuccess;
  if (ldc == N && count % 2 == 0 && aligned16(P) && (reinterpret_cast<uintptr_t>(C) & 7u) == 0) {
    finalize_kernel_2<<<grid_for(count / 2), kThreads, 0, stream>>>(P, count,
                                                                    reinterpret_cast<uint2*>(C));
  } else {
    finalize_kernel_1<<<grid_for(count), kThreads, 0, stream>>>(P, M, N,
                                                                reinterpret_cast<uint32_t*>(C), ldc);
  }
  note_launch();
  return cudaGetLastError();
}

}  // namespace det
