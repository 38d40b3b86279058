// Pipe-throughput microbenchmark: the roofline denominators for exact
// summation on the CUDA cores (integer ALU, integer multiply-add, FP64).
//
// Each thread keeps eight independent accumulators and updates them in a ring
// (accumulator i takes accumulator i+1 as an operand), so consecutive
// operations of one accumulator are separated by seven others and no two can
// be merged into one instruction.  Every operation is one inline-PTX
// instruction of the measured kind, its operands depend on run-time values,
// and the accumulators are folded into the output at the end, so none is
// removed.  The benchmark times a launch with CUDA events; the operation count
// is iters * 8 * (threads launched).
#include <cuda_runtime.h>
#include <stdint.h>

#include "det_gemm.h"
#include "det_kernels.h"

namespace det {
namespace {

constexpr int kChains = 8;
constexpr int kThreads = 256;

template <int kKind>
__global__ void __launch_bounds__(kThreads) pipe_kernel(int64_t iters, uint32_t seed, uint32_t* out) {
  const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  if (kKind == DET_PIPE_DFMA) {
    // x_i <- x_{i+1} * a + b: one fma per operation, converging to b / (1 - a)
    double x[kChains];
    const double a = 0.5 + 1e-9 * static_cast<double>(seed & 7u);
    const double b = 1.0 + 1e-12 * static_cast<double>(seed >> 3);
#pragma unroll
    for (int i = 0; i < kChains; ++i) x[i] = static_cast<double>(t + i);
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
      for (int i = 0; i < kChains; ++i)
        asm volatile("fma.rn.f64 %0, %1, %2, %3;" : "=d"(x[i]) : "d"(x[(i + 1) % kChains]), "d"(a), "d"(b));
    }
    double s = 0.0;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += x[i];
    out[t] = static_cast<uint32_t>(__double_as_longlong(s));
  } else if (kKind == DET_PIPE_FFMA) {
    float x[kChains];
    const float a = 0.5f + 1e-7f * static_cast<float>(seed & 7u);
    const float b = 1.0f + 1e-6f * static_cast<float>(seed >> 29);
#pragma unroll
    for (int i = 0; i < kChains; ++i) x[i] = static_cast<float>(t + i);
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
      for (int i = 0; i < kChains; ++i)
        asm volatile("fma.rn.f32 %0, %1, %2, %3;" : "=f"(x[i]) : "f"(x[(i + 1) % kChains]), "f"(a), "f"(b));
    }
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s ^= __float_as_uint(x[i]);
    out[t] = s;
  } else if (kKind == DET_PIPE_IMAD_WIDE) {
    uint64_t x[kChains];
    const uint32_t a = seed | 1u;
#pragma unroll
    for (int i = 0; i < kChains; ++i) x[i] = t + 977u * i;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
      for (int i = 0; i < kChains; ++i) {
        const uint32_t lo = static_cast<uint32_t>(x[(i + 1) % kChains]);
        asm volatile("mad.wide.u32 %0, %1, %2, %0;" : "+l"(x[i]) : "r"(lo), "r"(a));
      }
    }
    uint64_t s = 0;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s ^= x[i];
    out[t] = static_cast<uint32_t>(s ^ (s >> 32));
  } else {
    uint32_t x[kChains];
    const uint32_t a = seed | 1u, k = seed * 2654435761u;
#pragma unroll
    for (int i = 0; i < kChains; ++i) x[i] = t + 977u * i;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
      for (int i = 0; i < kChains; ++i) {
        const uint32_t y = x[(i + 1) % kChains];
        if (kKind == DET_PIPE_IADD)
          asm volatile("add.u32 %0, %0, %1;" : "+r"(x[i]) : "r"(y));
        else if (kKind == DET_PIPE_LOP3)
          asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(x[i]) : "r"(y), "r"(k));
        else
          asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(x[i]) : "r"(a), "r"(y));
      }
    }
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s ^= x[i];
    out[t] = s;
  }
}

}  // namespace
}  // namespace det

extern "C" det_status det_pipe_benchmark(int kind, int64_t iters, int64_t blocks, void* out,
                                         void* stream) {
  if (iters < 1 || blocks < 1 || blocks > (int64_t(1) << 20) || out == nullptr)
    return DET_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(out) & 3u) != 0) return DET_ERR_ALIGNMENT;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 grid(static_cast<unsigned>(blocks));
  uint32_t* o = static_cast<uint32_t*>(out);
  const uint32_t seed = 0x9E3779B9u ^ static_cast<uint32_t>(iters);
  switch (kind) {
    case DET_PIPE_IADD: det::pipe_kernel<DET_PIPE_IADD><<<grid, det::kThreads, 0, st>>>(iters, seed, o); break;
    case DET_PIPE_LOP3: det::pipe_kernel<DET_PIPE_LOP3><<<grid, det::kThreads, 0, st>>>(iters, seed, o); break;
    case DET_PIPE_IMAD: det::pipe_kernel<DET_PIPE_IMAD><<<grid, det::kThreads, 0, st>>>(iters, seed, o); break;
    case DET_PIPE_IMAD_WIDE:
      det::pipe_kernel<DET_PIPE_IMAD_WIDE><<<grid, det::kThreads, 0, st>>>(iters, seed, o);
      break;
    case DET_PIPE_FFMA: det::pipe_kernel<DET_PIPE_FFMA><<<grid, det::kThreads, 0, st>>>(iters, seed, o); break;
    case DET_PIPE_DFMA: det::pipe_kernel<DET_PIPE_DFMA><<<grid, det::kThreads, 0, st>>>(iters, seed, o); break;
    default: return DET_ERR_INVALID_ARG;
  }
  det::note_launch();
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

extern "C" int det_pipe_benchmark_ops_per_thread_iter(void) { return det::kChains; }
extern "C" int det_pipe_benchmark_threads_per_block(void) { return det::kThreads; }
