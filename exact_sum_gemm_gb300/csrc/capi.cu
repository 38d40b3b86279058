// C ABI of the exact-sum GEMM (declared in include/det_gemm.h).
//
// Validates every argument on the host and returns a det_status before
// anything is enqueued; then enqueues the kernels on the caller's stream.
// Nothing here allocates persistent memory, synchronises, or throws.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "det_gemm.h"
#include "det_gemm_internal.cuh"
#include "det_kernels.h"
#include "det_residue.cuh"

namespace det {
namespace {
std::atomic<uint64_t> g_launches{0};
}
void note_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }
}  // namespace det

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

det_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DET_OK : DET_ERR_CUDA; }

// Leading dimension rule: op 0 stores [rows, K] (ld >= K), op 1 stores [K, rows] (ld >= rows).
bool ld_ok(int64_t rows, int64_t K, int64_t ld, int op) {
  const int64_t need = op ? rows : K;
  return ld >= (need > 1 ? need : 1);
}

constexpr int64_t kMaxTiles = 0x7FFFFFFFll;

det_status validate_gemm(det_dtype dtype, int64_t M, int64_t N, int64_t K, const void* A,
                         int64_t lda, int opA, const void* B, int64_t ldb, int opB) {
  if (dtype != DET_F32 && dtype != DET_BF16) return DET_ERR_DTYPE;
  if (M < 0 || N < 0 || K < 0) return DET_ERR_SHAPE;
  if (K > DET_K_MAX) return DET_ERR_K_LIMIT;
  if (M > (int64_t(1) << 31) || N > (int64_t(1) << 31)) return DET_ERR_SHAPE;
  if (((M + 31) / 32) * ((N + 31) / 32) > kMaxTiles) return DET_ERR_SHAPE;
  if ((opA != 0 && opA != 1) || (opB != 0 && opB != 1)) return DET_ERR_INVALID_ARG;
  if (M > 0 && N > 0 && K > 0) {
    if (A == nullptr || B == nullptr) return DET_ERR_INVALID_ARG;
    if (!ld_ok(M, K, lda, opA) || !ld_ok(N, K, ldb, opB)) return DET_ERR_INVALID_ARG;
    const uintptr_t es = dtype == DET_F32 ? 4 : 2;
    if (!aligned(A, es) || !aligned(B, es)) return DET_ERR_ALIGNMENT;
  }
  return DET_OK;
}

std::atomic<int> g_batched_pipeline{1};          // det_set_batched_pipeline

det::GemmArgs make_args(det_dtype dtype, int64_t M, int64_t N, int64_t K, const void* A,
                        int64_t lda, int opA, const void* B, int64_t ldb, int opB) {
  det::GemmArgs a{};
  a.A = A;
  a.lda = lda;
  a.opA = opA;
  a.B = B;
  a.ldb = ldb;
  a.opB = opB;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bf16 = dtype == DET_BF16 ? 1 : 0;
  return a;
}

}  // namespace

extern "C" {

int det_abi_version(void) { return 1; }

int det_residue_moduli(det_dtype dtype, int64_t K) {
  if ((dtype != DET_F32 && dtype != DET_BF16) || K < 0 || K > DET_K_MAX) return -1;
  if (K == 0) return 0;
  det::GemmArgs a{};
  a.K = K;
  a.bf16 = dtype == DET_BF16 ? 1 : 0;
  return det::residue_planes_needed(a);
}

int det_moduli_used(int* out, int max) {
  if (max < 0) return -1;
  return det::moduli_record(out, max);
}

int det_set_wide_path(int enable) { return det::set_wide_path(enable); }

int det_set_batched_pipeline(int enable) { return g_batched_pipeline.exchange(enable ? 1 : 0); }

int det_tile_routes(int64_t* out) {
  if (out == nullptr) return -1;
  long long rec[4];
  if (det::route_record(rec) != 0) return -1;
  for (int i = 0; i < 4; ++i) out[i] = rec[i];
  return 0;
}

uint64_t det_kernel_launches(void) { return det::g_launches.load(std::memory_order_relaxed); }

const char* det_status_string(det_status s) {
  switch (s) {
    case DET_OK: return "DET_OK";
    case DET_ERR_INVALID_ARG: return "DET_ERR_INVALID_ARG: null pointer, bad op flag or leading dimension";
    case DET_ERR_DTYPE: return "DET_ERR_DTYPE: dtype must be DET_F32 or DET_BF16";
    case DET_ERR_SHAPE: return "DET_ERR_SHAPE: negative or too large size";
    case DET_ERR_K_LIMIT: return "DET_ERR_K_LIMIT: K exceeds 2^19 per GEMM call";
    case DET_ERR_OVERFLOW: return "DET_ERR_OVERFLOW: too many partials for int64 digit headroom";
    case DET_ERR_ALIGNMENT: return "DET_ERR_ALIGNMENT: pointer not aligned to its element size";
    case DET_ERR_CUDA: return "DET_ERR_CUDA: a CUDA call or kernel launch failed";
    case DET_ERR_NOALLOC_LIMIT:
      return "DET_ERR_NOALLOC_LIMIT: problem needs more scratch than det_gemm_partial_noalloc's "
             "fixed array (DET_NOALLOC_SCRATCH_BYTES)";
    case DET_ERR_TIMEOUT:
      return "DET_ERR_TIMEOUT: a bounded wait inside a kernel ran out; that call's outputs are NaN";
  }
  return "DET_ERR_UNKNOWN";
}

det_status det_release_scratch(void) { return from_cuda(det::pool_release()); }

det_status det_set_scratch_retention(uint64_t bytes) {
  return from_cuda(det::pool_set_retention(bytes));
}

det_status det_scratch_stats(uint64_t* allocations, uint64_t* reserved_bytes, uint64_t* used_bytes) {
  return from_cuda(det::pool_stats(allocations, reserved_bytes, used_bytes));
}

det_status det_gemm(det_dtype dtype, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                    int opA, const void* B, int64_t ldb, int opB, float* C, int64_t ldc,
                    void* stream) {
  det_status s = validate_gemm(dtype, M, N, K, A, lda, opA, B, ldb, opB);
  if (s != DET_OK) return s;
  if (M == 0 || N == 0) return DET_OK;
  if (C == nullptr || ldc < N) return DET_ERR_INVALID_ARG;
  if (!aligned(C, 4)) return DET_ERR_ALIGNMENT;
  det::GemmArgs a = make_args(dtype, M, N, K, A, lda, opA, B, ldb, opB);
  a.C = C;
  a.ldc = ldc;
  return from_cuda(det::launch_gemm(a, static_cast<cudaStream_t>(stream)));
}

det_status det_gemm_partial(det_dtype dtype, int64_t M, int64_t N, int64_t K, const void* A,
                            int64_t lda, int opA, const void* B, int64_t ldb, int opB, int64_t* P,
                            void* stream) {
  det_status s = validate_gemm(dtype, M, N, K, A, lda, opA, B, ldb, opB);
  if (s != DET_OK) return s;
  if (M == 0 || N == 0) return DET_OK;
  if (P == nullptr) return DET_ERR_INVALID_ARG;
  if (!aligned(P, 8)) return DET_ERR_ALIGNMENT;
  det::GemmArgs a = make_args(dtype, M, N, K, A, lda, opA, B, ldb, opB);
  a.P = P;
  return from_cuda(det::launch_gemm(a, static_cast<cudaStream_t>(stream)));
}

det_status det_gemm_partial_noalloc(det_dtype dtype, int64_t M, int64_t N, int64_t K,
                                    const void* A, int64_t lda, int opA, const void* B,
                                    int64_t ldb, int opB, int64_t* P, void* stream) {
  det_status s = validate_gemm(dtype, M, N, K, A, lda, opA, B, ldb, opB);
  if (s != DET_OK) return s;
  if (M == 0 || N == 0) return DET_OK;
  if (P == nullptr) return DET_ERR_INVALID_ARG;
  if (!aligned(P, 8)) return DET_ERR_ALIGNMENT;
  det::GemmArgs a = make_args(dtype, M, N, K, A, lda, opA, B, ldb, opB);
  a.P = P;
  if (!det::noalloc_fits(a)) return DET_ERR_NOALLOC_LIMIT;
  return from_cuda(det::launch_gemm_partial_noalloc(a, static_cast<cudaStream_t>(stream)));
}

det_status det_combine(int64_t M, int64_t N, const int64_t* const* parts, int n, int64_t* out,
                       void* stream) {
  if (M < 0 || N < 0) return DET_ERR_SHAPE;
  if (n < 1) return DET_ERR_SHAPE;
  if (n > DET_MAX_COMBINE) return DET_ERR_OVERFLOW;
  if (M > 0 && N > 0 && M > INT64_MAX / DET_PLANES / 8 / N) return DET_ERR_SHAPE;
  if (M == 0 || N == 0) return DET_OK;
  if (parts == nullptr || out == nullptr) return DET_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    if (parts[i] == nullptr) return DET_ERR_INVALID_ARG;
    if (!aligned(parts[i], 8)) return DET_ERR_ALIGNMENT;
  }
  if (!aligned(out, 8)) return DET_ERR_ALIGNMENT;
  return from_cuda(det::launch_combine(parts, n, M * N, out, static_cast<cudaStream_t>(stream)));
}

det_status det_finalize(int64_t M, int64_t N, const int64_t* P, float* C, int64_t ldc,
                        void* stream) {
  if (M < 0 || N < 0) return DET_ERR_SHAPE;
  if (M > 0 && N > 0 && M > INT64_MAX / DET_PLANES / 8 / N) return DET_ERR_SHAPE;
  if (M == 0 || N == 0) return DET_OK;
  if (P == nullptr || C == nullptr || ldc < N) return DET_ERR_INVALID_ARG;
  if (!aligned(P, 8) || !aligned(C, 4)) return DET_ERR_ALIGNMENT;
  return from_cuda(det::launch_finalize(P, M, N, C, ldc, static_cast<cudaStream_t>(stream)));
}

det_status det_linear_forward(det_dtype dtype, int64_t batch, int64_t in_features,
                              int64_t out_features, const void* x, const void* W, float* y,
                              void* stream) {
  // y[b,o] = sum_i x[b,i] W[o,i]: M = batch, N = out, K = in; both K-contiguous
  return det_gemm(dtype, batch, out_features, in_features, x, in_features, 0, W, in_features, 0,
                  y, out_features, stream);
}

det_status det_linear_dgrad(int64_t batch, int64_t in_features, int64_t out_features,
                            const float* dy, const float* W, float* dx, void* stream) {
  // dx[b,i] = sum_o dy[b,o] W[o,i]: M = batch, N = in, K = out; W read as [K, N]
  return det_gemm(DET_F32, batch, in_features, out_features, dy, out_features, 0, W, in_features,
                  1, dx, in_features, stream);
}

det_status det_linear_wgrad(int64_t batch, int64_t in_features, int64_t out_features,
                            const float* dy, const float* x, float* dW, void* stream) {
  // dW[o,i] = sum_b dy[b,o] x[b,i]: M = out, N = in, K = batch; both read as [K, rows]
  return det_gemm(DET_F32, out_features, in_features, batch, dy, out_features, 1, x, in_features,
                  1, dW, in_features, stream);
}

det_status det_gemm_strided_batched(det_dtype dtype, int64_t batch, int64_t M, int64_t N,
                                    int64_t K, const void* A, int64_t lda, int opA,
                                    int64_t strideA, const void* B, int64_t ldb, int opB,
                                    int64_t strideB, float* C, int64_t ldc, int64_t strideC,
                                    void* stream) {
  det_status s = validate_gemm(dtype, M, N, K, A, lda, opA, B, ldb, opB);
  if (s != DET_OK) return s;
  if (batch < 0 || strideA < 0 || strideB < 0 || strideC < 0) return DET_ERR_SHAPE;
  if (batch == 0 || M == 0 || N == 0) return DET_OK;
  if (C == nullptr || ldc < N) return DET_ERR_INVALID_ARG;
  if (!aligned(C, 4)) return DET_ERR_ALIGNMENT;
  const int64_t last = batch - 1;
  if ((strideA > 0 && last > INT64_MAX / 8 / strideA) || (strideB > 0 && last > INT64_MAX / 8 / strideB) ||
      (strideC > 0 && last > INT64_MAX / 8 / strideC))
    return DET_ERR_SHAPE;
  const int64_t es = dtype == DET_F32 ? 4 : 2;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // every entry in one residue-path pipeline where the shapes allow
  const int64_t kBig = int64_t(1) << 30;
  if (batch > 1 && g_batched_pipeline.load(std::memory_order_relaxed) != 0 && M <= kBig / batch &&
      N <= kBig / batch && strideA <= INT32_MAX && strideB <= INT32_MAX && strideC <= INT32_MAX) {
    det::GemmArgs g = make_args(dtype, batch * M, N, K, A, lda, opA, B, ldb, opB);
    g.C = C;
    g.ldc = ldc;
    g.batch = static_cast<int32_t>(batch);
    g.Me = static_cast<int32_t>(M);
    g.strideA = static_cast<int32_t>(strideA);
    g.strideB = static_cast<int32_t>(strideB);
    g.strideC = static_cast<int32_t>(strideC);
    if (det::batched_residue_ok(g)) return from_cuda(det::launch_gemm(g, st));
  }
  for (int64_t b = 0; b < batch; ++b) {
    const void* Ab = static_cast<const char*>(A) + b * strideA * es;
    const void* Bb = static_cast<const char*>(B) + b * strideB * es;
    det::GemmArgs a = make_args(dtype, M, N, K, Ab, lda, opA, Bb, ldb, opB);
    a.C = C + b * strideC;
    a.ldc = ldc;
    const det_status r = from_cuda(det::launch_gemm(a, st));
    if (r != DET_OK) return r;
  }
  return DET_OK;
}

det_status det_linear_forward_bias(det_dtype dtype, int64_t batch, int64_t in_features,
                                   int64_t out_features, const void* x, const void* W,
                                   const void* bias, float* y, void* stream) {
  if (bias == nullptr)
    return det_linear_forward(dtype, batch, in_features, out_features, x, W, y, stream);
  if (in_features < 0 || in_features + 1 > DET_K_MAX) return in_features < 0 ? DET_ERR_SHAPE
                                                                             : DET_ERR_K_LIMIT;
  det_status s = validate_gemm(dtype, batch, out_features, in_features + 1, x, in_features + 1 > 1
                               ? in_features + 1 : 1, 0, W, in_features + 1, 0);
  if (s != DET_OK) return s;
  if (batch == 0 || out_features == 0) return DET_OK;
  if (x == nullptr || W == nullptr || y == nullptr) return DET_ERR_INVALID_ARG;
  const uintptr_t es = dtype == DET_F32 ? 4 : 2;
  if (!aligned(bias, es) || !aligned(y, 4)) return DET_ERR_ALIGNMENT;
  return from_cuda(det::launch_linear_bias(dtype == DET_BF16 ? 1 : 0, batch, in_features,
                                           out_features, x, W, bias, y,
                                           static_cast<cudaStream_t>(stream)));
}

det_status det_linear_bias_grad(int64_t batch, int64_t out_features, const float* dy, float* db,
                                void* stream) {
  if (batch < 0 || out_features < 0) return DET_ERR_SHAPE;
  if (batch > DET_K_MAX) return DET_ERR_K_LIMIT;
  if (out_features > (int64_t(1) << 31)) return DET_ERR_SHAPE;
  if (out_features == 0) return DET_OK;
  if (db == nullptr || (batch > 0 && dy == nullptr)) return DET_ERR_INVALID_ARG;
  if (!aligned(db, 4) || !aligned(dy, 4)) return DET_ERR_ALIGNMENT;
  return from_cuda(det::launch_bias_grad(batch, out_features, dy, db,
                                         static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
