// DetLinear extras: an exact bias term and its exact gradient.
//
// The bias is one more product of the sum: y[r,o] = RNE_f32(sum_i x[r,i]
// W[o,i] + 1 * bias[o]), so it goes through the same exact accumulation and
// the same single rounding as every other product.  The operands are widened
// by one K column, [x | 1] and [W | bias], in pool scratch by a copy kernel,
// and the widened GEMM is an ordinary det_gemm.  The bias gradient
// db[o] = sum_r dy[r,o] is the exact GEMM of a row of ones with dy read as
// [out, rows] (no transpose materialised).
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstring>

#include "det_kernels.h"

namespace det {
namespace {

constexpr int kThreads = 256;

// dst [rows, in + 1] = [src | value_r]: value_r = col[r] if col, else `one`.
template <typename T>
__global__ void __launch_bounds__(kThreads) widen_kernel(const T* src, int64_t rows, int64_t in,
                                                          const T* col, T one, T* dst) {
  const int64_t w = in + 1;
  const int64_t total = rows * w;
  for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * kThreads) {
    const int64_t r = i / w, k = i - r * w;
    dst[i] = k < in ? src[r * in + k] : (col ? col[r] : one);
  }
}

__global__ void __launch_bounds__(kThreads) ones_kernel(float* p, int64_t n) {
  for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * kThreads)
    p[i] = 1.0f;
}

unsigned grid_for(int64_t n) {
  const int64_t g = (n + kThreads - 1) / kThreads;
  return static_cast<unsigned>(g < 4096 ? (g > 0 ? g : 1) : 4096);
}

template <typename T>
cudaError_t widen(const void* src, int64_t rows, int64_t in, const void* col, uint32_t one_bits,
                  void* dst, cudaStream_t stream) {
  T one;
  static_assert(sizeof(T) <= sizeof(uint32_t), "16- or 32-bit elements");
  std::memcpy(&one, &one_bits, sizeof(T));
  widen_kernel<T><<<grid_for(rows * (in + 1)), kThreads, 0, stream>>>(
      static_cast<const T*>(src), rows, in, static_cast<const T*>(col), one, static_cast<T*>(dst));
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_linear_bias(int bf16, int64_t rows, int64_t in, int64_t out, const void* x,
                               const void* W, const void* bias, float* y, cudaStream_t stream) {
  if (rows == 0 || out == 0) return cudaSuccess;
  const size_t es = bf16 ? 2 : 4;
  const size_t xb = (size_t(rows) * (in + 1) * es + 255) / 256 * 256;
  const size_t wb = size_t(out) * (in + 1) * es;
  void* scratch = nullptr;
  cudaError_t e = pool_alloc(&scratch, xb + wb, stream);
  if (e != cudaSuccess) return e;
  void* xw = scratch;
  void* ww = static_cast<char*>(scratch) + xb;
  // 1.0 as a binary32 pattern, or its top half for bf16 (exact)
  if (bf16) {
    e = widen<uint16_t>(x, rows, in, nullptr, 0x3F80u, xw, stream);
    if (e == cudaSuccess) e = widen<uint16_t>(W, out, in, bias, 0u, ww, stream);
  } else {
    e = widen<uint32_t>(x, rows, in, nullptr, 0x3F800000u, xw, stream);
    if (e == cudaSuccess) e = widen<uint32_t>(W, out, in, bias, 0u, ww, stream);
  }
  if (e == cudaSuccess) {
    GemmArgs a{};
    a.A = xw;
    a.lda = in + 1;
    a.opA = 0;
    a.B = ww;
    a.ldb = in + 1;
    a.opB = 0;
    a.M = rows;
    a.N = out;
    a.K = in + 1;
    a.bf16 = bf16;
    a.C = y;
    a.ldc = out;
    e = launch_gemm(a, stream);
  }
  const cudaError_t f = cudaFreeAsync(scratch, stream);
  return e != cudaSuccess ? e : f;
}

cudaError_t launch_bias_grad(int64_t rows, int64_t out, const float* dy, float* db,
                             cudaStream_t stream) {
  if (out == 0) return cudaSuccess;
  void* ones = nullptr;
  cudaError_t e = pool_alloc(&ones, sizeof(float) * size_t(rows > 0 ? rows : 1), stream);
  if (e != cudaSuccess) return e;
  ones_kernel<<<grid_for(rows), kThreads, 0, stream>>>(static_cast<float*>(ones), rows);
  note_launch();
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    // [1, out] = ones [1, rows] x dy^T, with dy read as B [out, rows] stored [rows, out] (op 1)
    GemmArgs a{};
    a.A = ones;
    a.lda = rows > 0 ? rows : 1;
    a.opA = 0;
    a.B = dy;
    a.ldb = out;
    a.opB = 1;
    a.M = 1;
    a.N = out;
    a.K = rows;
    a.bf16 = 0;
    a.C = db;
    a.ldc = out;
    e = launch_gemm(a, stream);
  }
  const cudaError_t f = cudaFreeAsync(ones, stream);
  return e != cudaSuccess ? e : f;
}

}  // namespace det
