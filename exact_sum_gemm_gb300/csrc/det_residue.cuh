// Moduli and launch plumbing of the residue (CRT) decomposition.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "det_kernels.h"

namespace det {

// Odd, pairwise coprime moduli <= 255: balanced residues lie in [-127, 127]
// (exact in bf16), products of two in [-16129, 16129], and 1024 such products
// plus a reduced carry stay below 2^24, where fp32 accumulation is exact.
// The product of all 14 exceeds 2^109, enough for |S| < 2^19 * 2^86 * 2
// (f32 shallow integers are below 2^(24+19)).
constexpr int kNumModuli = 14;
__host__ __device__ constexpr int modulus(int i) {
  return i == 0 ? 255 : i == 1 ? 253 : i == 2 ? 251 : i == 3 ? 247 : i == 4 ? 241 : i == 5 ? 239
       : i == 6 ? 233 : i == 7 ? 229 : i == 8 ? 227 : i == 9 ? 223 : i == 10 ? 217 : i == 11 ? 211
       : i == 12 ? 199 : 197;
}
// (p_0 * ... * p_{i-1})^{-1} mod p_i, for Garner's CRT (compile-time use).
__host__ __device__ constexpr int garner_inverse(int i) {
  int prod = 1;
  for (int j = 0; j < i; ++j) prod = (prod * (modulus(j) % modulus(i))) % modulus(i);
  for (int c = 1; c < modulus(i); ++c)
    if ((prod * c) % modulus(i) == 1) return c;
  return 1;
}

constexpr int kChunkK = 1024;     // K per exact fp32 accumulation window
constexpr int kStageK = 64;       // K per TMA/MMA stage (one 128-byte swizzle row of bf16)

struct ResidueOperand {
  const void* X;
  int64_t ld;
  int op;
  int64_t rows;
  int64_t K;
  int64_t Kp;                 // K rounded up to kStageK (zero padded)
  const int* emax;            // [rows]
  __nv_bfloat16* planes;      // [nplanes][rows][Kp]
  int* list_count;            // [rows], zeroed before the launch
  uint2* list;                // [rows][cap]: (k, raw bits) of deep / non-finite elements
  int cap;
};

struct ReconArgs {
  const uint8_t* res;         // [nplanes][M][N] residues in [0, p_i)
  int nplanes;
  const int* emaxA;
  const int* emaxB;
  const uint8_t* route;       // 64x64 tiles: 1 = general kernel (skipped here)
  const int* countA;
  const uint2* listA;
  const int* countB;
  const uint2* listB;
  int cap;
  const int* error;           // nonzero: the tensor-core kernel gave up (outputs NaN)
};

int residue_planes_needed(const GemmArgs& g);
cudaError_t launch_residues(const ResidueOperand& o, int bf16, int nplanes, cudaStream_t stream);
// deep_lists: scratch of M + N ints; deep_counters: 2 ints, zero at launch.
cudaError_t launch_reconstruct(const GemmArgs& g, const ReconArgs& ra, int* deep_lists,
                               int* deep_counters, cudaStream_t stream);

struct ResGemmArgs {
  const __nv_bfloat16* A;     // [nplanes][M][Kp]
  const __nv_bfloat16* B;     // [nplanes][N][Kp]
  int64_t M, N, Kp;
  int nplanes;
  uint8_t* res;               // [nplanes][M][N]
  int* error;
};
cudaError_t launch_residue_gemm(const ResGemmArgs& a, cudaStream_t stream);

}  // namespace det
