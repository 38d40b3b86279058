// Internal launch interface between the C ABI (capi.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace det {

// Devices a process may use this library on (per-device state is kept in
// arrays of this size).
constexpr int kMaxDevices = 64;

// One-time set-up per device: run(init) calls init(dev) with the current
// device `dev`, once per device and under a lock, until it succeeds.  Function
// attributes (cudaFuncSetAttribute) belong to the device that was current when
// they were set, so they are configured through one of these.
class PerDeviceOnce {
 public:
  template <class F>
  cudaError_t run(F&& init) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev]) return cudaSuccess;
    e = init(dev);
    if (e == cudaSuccess) done_[dev] = true;
    return e;
  }

 private:
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
};

// Sticky device-side status word of this library on the current device
// (bit kStatusTimeout: a bounded wait in one of its kernels ran out).  The
// address is looked up once per device.
constexpr unsigned kStatusTimeout = 1u;
cudaError_t device_status_word(unsigned** out);

// Count one enqueued kernel (diagnostic; see det_kernel_launches).
void note_launch(int n = 1);

// Stages timed by det_stage_timing / det_stage_report.
enum Stage { kStagePrepass = 0, kStageResiduePlanes, kStageResidueGemm, kStageReconstruct,
             kStageGeneral, kStageBand, kStageWideStats, kStageWidePlanes, kStageWideGemm,
             kStageWideReconstruct, kNumStages };

// Records a CUDA event pair around its scope on `stream` while stage timing is on.
class StageScope {
 public:
  StageScope(int stage, cudaStream_t stream);
  ~StageScope();
  StageScope(const StageScope&) = delete;
  StageScope& operator=(const StageScope&) = delete;

 private:
  int stage_;
  cudaStream_t stream_;
  cudaEvent_t start_{}, stop_{};
  bool active_ = false;
};

struct GemmArgs {
  const void* A;
  int64_t lda;
  int opA;            // 0: element (m,k) at A[m*lda+k]; 1: at A[k*lda+m]
  const void* B;
  int64_t ldb;
  int opB;            // 0: element (n,k) at B[n*ldb+k]; 1: at B[k*ldb+n]
  int64_t M, N, K;
  int bf16;           // operand dtype: 0 = f32, 1 = bf16
  float* C;           // fused-finalize output (det_gemm), or null
  int64_t ldc;
  int64_t* P;         // canonical digit planes [20][M][N] (det_gemm_partial), or null
  // A strided batch computed as one problem (det_gemm_strided_batched, C
  // output only): `batch` entries of Me rows each are stacked as the
  // M = batch * Me rows of A and C; output row m belongs to entry
  // e = m / Me, whose A, B and C start e * strideA, e * strideB elements and
  // e * strideC floats after entry 0's.  Per-row arrays of B hold every
  // entry's N rows, stacked: row n of entry e at e * N + n.  batch = 1: a
  // plain GEMM (Me and the strides unused).  32-bit fields (the batched path
  // takes stacked row counts below 2^30 and strides below 2^31): the kernels
  // that take GemmArgs by value keep their register allocation.
  int32_t batch = 1;
  int32_t Me = 0;
  int32_t strideA = 0, strideB = 0, strideC = 0;
};

// Quotient of row indices of a strided batch (below 2^30: a 32-bit division).
__host__ __device__ inline int64_t entry_div(int64_t r, int64_t rows) {
  return static_cast<int64_t>(static_cast<uint32_t>(r) / static_cast<uint32_t>(rows));
}
// Rows of B's per-row arrays (every entry's N rows).
__host__ __device__ inline int64_t rows_of_b(const GemmArgs& g) {
  return g.batch > 1 ? g.batch * g.N : g.N;
}
// B's stacked row for output row m, column n.
__host__ __device__ inline int64_t brow_of(const GemmArgs& g, int64_t m, int64_t n) {
  return g.batch > 1 ? entry_div(m, g.Me) * g.N + n : n;
}
// Element offsets of A's (m, k) and of B's stacked row s at k.
__host__ __device__ inline int64_t a_offset(const GemmArgs& g, int64_t m, int64_t k) {
  int64_t e = 0;
  if (g.batch > 1) {
    e = entry_div(m, g.Me);
    m -= e * g.Me;
  }
  return e * int64_t(g.strideA) + (g.opA ? k * g.lda + m : m * g.lda + k);
}
__host__ __device__ inline int64_t b_offset(const GemmArgs& g, int64_t s, int64_t k) {
  int64_t e = 0;
  if (g.batch > 1) {
    e = entry_div(s, g.N);
    s -= e * g.N;
  }
  return e * int64_t(g.strideB) + (g.opB ? k * g.ldb + s : s * g.ldb + k);
}
// Offset (in floats) of C's output row m.
__host__ __device__ inline int64_t c_row_offset(const GemmArgs& g, int64_t m) {
  if (g.batch <= 1) return m * g.ldc;
  const int64_t e = entry_div(m, g.Me);
  return e * int64_t(g.strideC) + (m - e * g.Me) * g.ldc;
}

// Wide residue path on (1, the default) or off (0); returns the previous setting.
int set_wide_path(int enable);

// Exact GEMM; writes C (if args.C) or the digit planes P (if args.P).  A
// strided batch (batch > 1) must pass batched_residue_ok.
cudaError_t launch_gemm(const GemmArgs& args, cudaStream_t stream);
// Whether a strided batch can run as one residue-path problem: C output,
// K-contiguous operands whose rows suit the fused planes kernel, N and the
// entries' rows multiples of 64.
bool batched_residue_ok(const GemmArgs& args);

// Stream-ordered scratch from the library's memory pool (one per device, kept
// reserved between calls); release with cudaFreeAsync on the same stream.
cudaError_t pool_alloc(void** p, size_t bytes, cudaStream_t stream);
// Allocations taken so far (all devices) and the current device's pool's
// reserved and used bytes (0 before its first allocation).
cudaError_t pool_stats(uint64_t* allocations, uint64_t* reserved, uint64_t* used);
// Synchronise the current device, then return its pool's unused memory.
cudaError_t pool_release();
// Bytes every pool keeps reserved after its frees (default: all of them).
cudaError_t pool_set_retention(uint64_t bytes);

// y = RNE_f32(x W^T + bias): the bias enters as one more exact product,
// 1 * bias[o], through [x | 1] and [W | bias] built in pool scratch.
// x [rows, in], W [out, in], bias [out] contiguous, all of one dtype.
cudaError_t launch_linear_bias(int bf16, int64_t rows, int64_t in, int64_t out, const void* x,
                               const void* W, const void* bias, float* y, cudaStream_t stream);

// db[o] = RNE_f32(sum_r dy[r, o]) exactly (dy fp32 [rows, out]).
cudaError_t launch_bias_grad(int64_t rows, int64_t out, const float* dy, float* db,
                             cudaStream_t stream);

constexpr int kMaxPartsPerLaunch = 16;

// out = canonical(sum of parts), over count = M*N outputs of 20 planes each.
cudaError_t launch_combine(const int64_t* const* parts, int n, int64_t count, int64_t* out,
                           cudaStream_t stream);

// C[m*ldc+n] = RNE_f32(value of P[:, m, n]).
cudaError_t launch_finalize(const int64_t* P, int64_t M, int64_t N, float* C, int64_t ldc,
                            cudaStream_t stream);

}  // namespace det
