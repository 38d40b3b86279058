// Moduli and launch plumbing of the residue (CRT) decomposition.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "det_kernels.h"

namespace det {

// Odd, pairwise coprime moduli in [197, 255].  The operand planes hold
// residues r with |r| <= 138 (nearly balanced, exact in bf16, which holds
// integers up to 256), so a product of two is at most 138^2 = 19044 in
// magnitude, and 832 such products plus a reduced carry (< 131) stay below
// 2^24, where fp32 accumulation is exact.  The product of all 14 moduli
// exceeds 2^109, enough for |S| < 2^19 * 2^84 * 2 (1 + 2^-7) (f32 shallow
// integers are below 2^(24+18)).
//
// The wide path (wide.cu) continues the list with 2^8 and 25 primes from 193
// down to 71, all coprime to the first 14 and to one another: 40 moduli whose
// product exceeds 2^292.  2^8 is even, but its reduction below rounds a/256
// exactly (1/256 is exact in binary32), so its residues are the nearest
// ones, |r| <= 128.
constexpr int kNumModuli = 14;
constexpr int kNumModuliWide = 40;
__host__ __device__ constexpr int modulus(int i) {
  return i == 0 ? 255 : i == 1 ? 253 : i == 2 ? 251 : i == 3 ? 247 : i == 4 ? 241 : i == 5 ? 239
       : i == 6 ? 233 : i == 7 ? 229 : i == 8 ? 227 : i == 9 ? 223 : i == 10 ? 217 : i == 11 ? 211
       : i == 12 ? 199 : i == 13 ? 197 : i == 14 ? 256 : i == 15 ? 193 : i == 16 ? 191
       : i == 17 ? 181 : i == 18 ? 179 : i == 19 ? 173 : i == 20 ? 167 : i == 21 ? 163
       : i == 22 ? 157 : i == 23 ? 151 : i == 24 ? 149 : i == 25 ? 139 : i == 26 ? 137
       : i == 27 ? 131 : i == 28 ? 127 : i == 29 ? 113 : i == 30 ? 109 : i == 31 ? 107
       : i == 32 ? 103 : i == 33 ? 101 : i == 34 ? 97 : i == 35 ? 89 : i == 36 ? 83
       : i == 37 ? 79 : i == 38 ? 73 : 71;
}
// Balanced representatives, inverses and products modulo the moduli (compile
// time).
__host__ __device__ constexpr int balanced_rep(long long x, int p) {
  long long r = x % p;
  if (r < 0) r += p;
  return static_cast<int>(r > (p - 1) / 2 ? r - p : r);
}
__host__ __device__ constexpr int inverse_mod(int a, int p) {
  for (int c = 1; c < p; ++c)
    if ((a * c) % p == 1) return c;
  return 0;
}
// Exact modular reduction in binary32 (integers below 2^24 are exact there,
// and the fp32 FMA pipes outrun the integer multiplier).  For an integer-
// valued a with |a| <= 2^26 and an odd modulus p in [197, 255], with
// inv_p = 1/p to within one ulp (so |a * inv_p| < 2^19, where adding
// 1.5*2^23 rounds to an integer):
//   q = (a * inv_p + 1.5*2^23) - 1.5*2^23      (one rounding to an integer)
//   r = a - q * p                               (one fma: exact, r is small)
// Before rounding, q is within |a|/p * 2^-23 of the real a/p.  a/p is never
// a half-integer (p is odd) and a non-integer a/p lies at least 1/(2p) > 2^-9
// from one; so whenever |a| < 2^14 * p the rounding gives the nearest integer
// and r is the balanced residue in [-(p-1)/2, (p-1)/2].  Otherwise q may be
// one off: |r| <= p * (1/2 + |a|/p * 2^-23), which is below 131 for
// |a| <= 2^24 and below 139 for |a| <= 2^26.  A zero result is +0 unless a
// is -0.
constexpr float kRoundMagic = 12582912.0f;           // 1.5 * 2^23

__device__ __forceinline__ float near_mod_f32(float a, float p, float inv_p) {
  const float q = __fsub_rn(__fmaf_rn(a, inv_p, kRoundMagic), kRoundMagic);
  return __fmaf_rn(-q, p, a);
}

constexpr int kChunkK = 832;      // K per exact fp32 accumulation window (13 stages)
constexpr int kStageK = 64;       // K per TMA/MMA stage (one 128-byte swizzle row of bf16)
static_assert(kChunkK % kStageK == 0, "accumulation windows are whole stages");
static_assert(int64_t(kChunkK) * 138 * 138 + 131 < (int64_t(1) << 24), "window stays exact in fp32");

// Plane layout.  Rows are taken in groups of kPlaneRows; for each group and
// 64-k stage the nplanes planes follow one another, each a 32 x 64 bf16 block
// (4 KB, 128 bytes per row):
//   plane u of element (r, k) at
//   (((r / 32) * Kp/64 + k / 64) * nplanes + u) * 2048 + (r % 32) * 64 + k % 64.
// The residue kernel writes an element pair's planes at fixed 4 KB steps, and
// one modulus's stage for 32 rows is one contiguous 4 KB block for the TMA.
// Padding rows (up to a multiple of 32) hold zero residues.
constexpr int kPlaneRows = 32;
inline int64_t plane_rows(int64_t rows) { return (rows + kPlaneRows - 1) / kPlaneRows * kPlaneRows; }

struct ResidueOperand {
  const void* X;
  int64_t ld;
  int op;
  int32_t group_rows = 0;     // > 0: the rows are groups of group_rows (a strided batch's
                              //   entries), group g starting g * group_stride elements on
                              //   (both 32-bit and in padding: the operand keeps its size)
  int64_t rows;
  int64_t K;
  int64_t Kp;                 // K rounded up to kStageK (zero padded)
  int* emax;                  // [rows] (written by the fused kernel, read by the others)
  __nv_bfloat16* planes;      // [rows/32][Kp/64][nplanes][32][64] (rows padded to 32, see
                              // kPlaneRows)
  int* list_count;            // [rows], zeroed before the launch
  uint2* list;                // [rows][cap]: (k, raw bits) of deep / non-finite elements
  int cap;
  int32_t group_stride = 0;
  unsigned long long* norm;   // [rows], zeroed before the launch: an upper bound of
                              // sum_k X_int^2 / 2^norm_shift over the row's shallow elements
  unsigned* keymax;           // fused kernel: [rows], zeroed (row maxima of exponent keys)
  unsigned long long* norm_max;  // fused kernel: zeroed slot for the largest norm of these rows
  unsigned* dmax;             // fused kernel: [rows/64], zeroed: largest deep count of each
                              //   64-row block (or null)
};
static_assert(sizeof(ResidueOperand) == 15 * 8, "the group fields sit in padding");

// Element offset of an operand's row r (K-contiguous or not).
__host__ __device__ inline int64_t operand_row_offset(const ResidueOperand& o, int64_t r) {
  if (o.group_rows <= 0) return r * o.ld;
  const int64_t g = entry_div(r, o.group_rows);      // grouped rows stay below 2^30
  return g * int64_t(o.group_stride) + (r - g * o.group_rows) * o.ld;
}

// Thresholds of the moduli choice: P moduli suffice for a row band whose
// largest row-norm bounds are a (A) and b (B) when the 128-bit a * b is below
// t[P] = (hi[P], lo[P]), an integer no larger than
//   prod_P^2 / (2^(2 norm_shift + 2) (1 + 2^-7)^2 (1 + 2^-29)),
// so that prod_P > 2 (1 + 2^-7) sqrt(a b) 2^norm_shift >= 2 (1 + 2^-7) |S|.
struct ModuliThresholds {
  unsigned long long hi[kNumModuli + 1];
  unsigned long long lo[kNumModuli + 1];
};
ModuliThresholds moduli_thresholds(int bf16);
__device__ __forceinline__ int choose_moduli(unsigned long long a, unsigned long long b, int least,
                                             int most, const ModuliThresholds& t) {
  const unsigned long long phi = __umul64hi(a, b), plo = a * b;
  for (int P = least; P < most; ++P)
    if (phi < t.hi[P] || (phi == t.hi[P] && plo < t.lo[P])) return P;
  return most;
}

// The fewest moduli with compiled kernels (f32 12, bf16 8).
__host__ __device__ constexpr int planes_least(int bf16) { return bf16 ? 8 : 12; }

// Row norms are summed in units of 2^norm_shift (f32: |X_int| < 2^42, so a
// row of K <= 2^19 sums below 2^51 units; bf16: |X_int| < 2^26, below 2^55).
__host__ __device__ constexpr int norm_shift(int bf16) { return bf16 ? 16 : 52; }

struct ReconArgs {
  const int8_t* res;          // [nplanes][M][N] balanced residues, |r| <= (p_i - 1) / 2
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
  int64_t m_begin, m_end;     // rows of C handled by this launch (a band)
  const int* used;            // moduli this band uses (device int, <= nplanes), or null
};

// Moduli the worst case of this dtype and K needs (the planes are written for
// this many), and the fewest a band may use (compiled kernel counts).
int residue_planes_needed(const GemmArgs& g);
int residue_planes_least(int bf16);
// Diagnostic: the counts the last residue-path call chose, one per row band
// (copied from device memory: synchronises with the device).  Returns the
// number written (at most max), or -1 on a CUDA error.
int moduli_record(int* out, int max);
void note_moduli_bands(int bands);
// The fused path for K-contiguous, vector-aligned operands with K <= kFusedK:
// one launch per row band computes the rows' exponent maxima, deep lists,
// residue planes and norm bounds (no separate exponent pre-pass), and its
// last block writes the band's moduli count.  maxA / maxB: the zeroed slots
// of the band's A rows and of B's rows (B's filled by band 0's launch, which
// also covers B); done: a zeroed block counter per launch.
constexpr int kFusedK = 4096;
// A band whose every 64x64 tile goes to the general tiles (the smallest
// 64-row-block maximum of deep counts of its rows of A plus that of B's rows
// exceeds the lists' capacity) computes no modulus: its count is 0 and its
// tensor-core GEMM returns at once; the routing sends all its tiles on.
struct FusedBand {
  const unsigned long long* maxA;
  const unsigned long long* maxB;
  unsigned* done;
  int* used;
  int band, least, most;
  ModuliThresholds thr;
  const unsigned* dmaxA;      // the band's 64-row blocks of A (null: never skip)
  int64_t blocksA;
  const unsigned* dmaxB;      // B's 64-row blocks
  int64_t blocksB;
  int cap;
};
bool fused_residues_ok(const ResidueOperand& o, int bf16);
// Band 0 with B (o1 null: a band b >= 1 alone).
cudaError_t launch_residues_fused(const ResidueOperand& o0, const ResidueOperand* o1, int bf16,
                                  int nplanes, const FusedBand& fb, cudaStream_t stream);
// One block: the moduli count of a row band, the smallest in [least, most]
// whose product exceeds 2 (1 + 2^-7) sqrt(max normA * max normB) 2^shift,
// written to *used (a Cauchy-Schwarz bound of every |S| in the band).
// maxima: two zeroed 8-byte slots of scratch per launch.
// countA / countB (the rows' deep counts) and cap: as FusedBand, a band all of
// whose tiles go to the general tiles gets the count 0 (null countA: never).
cudaError_t launch_moduli(const unsigned long long* normA, int64_t rowsA,
                          const unsigned long long* normB, int64_t rowsB, int bf16, int least,
                          int most, int* used, int band, unsigned long long* maxima,
                          const int* countA, const int* countB, int cap, cudaStream_t stream);
cudaError_t launch_residues(const ResidueOperand& o, int bf16, int nplanes, cudaStream_t stream);
// Two operands' planes in one launch (one grid covering both).
cudaError_t launch_residues2(const ResidueOperand& o0, const ResidueOperand& o1, int bf16, int nplanes,
                             cudaStream_t stream);
// The outputs of a band whose row of A and column of B hold no deep element.
// For det_gemm_partial (g.P set) the launch may write whole row segments of
// digit planes, placeholder zeros in the deep columns included: the band's
// deep kernel must then run after it (it does not touch deep rows or the
// general tiles).
cudaError_t launch_reconstruct_fast(const GemmArgs& g, const ReconArgs& ra, cudaStream_t stream);
// The band's other outputs: those of its deep rows (kDeepRows) and of its
// deep columns outside deep rows (kDeepCols).  For det_gemm both kernels may
// run at once; for det_gemm_partial the deep-column part follows the fast
// kernel.  deep_lists: the rows of A then the columns of C that hold deep
// elements (M + N ints), with their two counts in deep_counters, as the
// routing step lists them.  blocks_per_sm: 1, or 2 where nothing else is
// meant to run beside it.
constexpr int kDeepRows = 1, kDeepCols = 2;
cudaError_t launch_reconstruct_deep(const GemmArgs& g, const ReconArgs& ra, int* deep_lists,
                                    int* deep_counters, int parts, int blocks_per_sm,
                                    cudaStream_t stream);

struct ResGemmArgs {
  const __nv_bfloat16* A;     // [M/32][Kp/64][nplanes][32][64] (ResidueOperand::planes)
  const __nv_bfloat16* B;     // [N/32][Kp/64][nplanes][32][64]
  int64_t M, N, Kp;
  int nplanes;
  int8_t* res;                // [nplanes][.][N] balanced residues: plane u of row m at
  int64_t res_plane;          //   res + u * res_plane + m * N
  int* error;                 // per-call flag: a bounded wait ran out (outputs become NaN)
  unsigned* status;           // the library's sticky device status word, or null
  const int* used;            // moduli to compute (device int, in [used_min, nplanes]; 0:
  int used_min;               //   nothing), or null for all nplanes; the grid is sized for used_min
  int grid_moduli;            // if > 0: size the grid for this many moduli instead
  // A strided batch's band (entry_rows > 0): M = whole entries of entry_rows
  // rows, the first being entry entry0; output rows of local entry e take
  // B's planes rows (entry0 + e) * N + n.  Only each entry's own tiles are
  // computed; rows and columns past the entry's are not written.
  int64_t entry_rows = 0;
  int64_t entry0 = 0;
  // (plain tiling only) a device list of the output tiles to compute, count
  // first, as tile indices of the launch's own tiling (row-major over the
  // whole M x N); null: every tile
  const int* tile_list = nullptr;
};
cudaError_t launch_residue_gemm(const ResGemmArgs& a, cudaStream_t stream);

// Rows of B's planes a launch reads (every entry's up to its band's last).
__host__ __device__ inline int64_t gemm_b_rows(const ResGemmArgs& a) {
  return a.entry_rows > 0 ? (a.entry0 + a.M / a.entry_rows) * a.N : a.N;
}
// How a launch enumerates its output tiles: every tile of M x N, each
// strided-batch entry's own (entry_rows > 0), or a device-side list
// (tile_list).  Each is its own compiled variant of the tensor-core kernels,
// so the plain one keeps its register allocation.
constexpr int kTilingPlain = 0, kTilingEntries = 1, kTilingListed = 2;
__host__ __device__ inline int tiling_of(const ResGemmArgs& a) {
  return a.entry_rows > 0 ? kTilingEntries : (a.tile_list != nullptr ? kTilingListed : kTilingPlain);
}
// Entries a TM x TN tile packs (a strided batch whose entries' rows and
// columns both divide the tile's): tile k takes entries kG .. kG + G - 1, A's
// rows and B's rows of those entries side by side, and only the diagonal
// blocks (an entry's rows with its own columns) are outputs.  1: one entry
// per tile.
template <int TM, int TN, int kTiling>
__host__ __device__ inline int64_t gemm_pack(const ResGemmArgs& a) {
  if (kTiling != kTilingEntries || a.entry_rows <= 0 || a.entry_rows > TM || a.N > TN ||
      TM % a.entry_rows != 0 || TN % a.N != 0)
    return 1;
  const int64_t gm = TM / a.entry_rows, gn = TN / a.N;
  return gm < gn ? gm : gn;
}
// Output tiles of TM x TN of a launch: the whole M x N (also the bound of a
// listed launch, whose own count is on the device), or each entry's own
// (pack entries per tile where they fit).
template <int TM, int TN, int kTiling>
__host__ __device__ inline int64_t gemm_tiles(const ResGemmArgs& a, int64_t pack) {
  const int64_t tn = (a.N + TN - 1) / TN;
  if (kTiling != kTilingEntries || a.entry_rows <= 0) return ((a.M + TM - 1) / TM) * tn;
  const int64_t entries = a.M / a.entry_rows;
  if (pack > 1) return (entries + pack - 1) / pack;
  return entries * ((a.entry_rows + TM - 1) / TM) * tn;
}
// Tile t: its first row of A (in the launch), first row of B's planes, first
// output column, and the end of its rows' entry (rows from there on are
// another entry's, or past M: computed but not written).  A packed tile's
// first column is 0 and m_end the end of its last entry; a listed launch's
// t-th tile is the list's t-th entry.
template <int TM, int TN, int kTiling>
__host__ __device__ inline void gemm_tile(const ResGemmArgs& a, int64_t pack, int64_t t, int64_t& m0,
                                          int64_t& nb0, int64_t& n0, int64_t& m_end) {
  const int64_t tn = (a.N + TN - 1) / TN;
  if (kTiling == kTilingEntries && a.entry_rows > 0 && pack > 1) {
    m0 = t * pack * a.entry_rows;
    n0 = 0;
    nb0 = (a.entry0 + t * pack) * a.N;
    m_end = m0 + pack * a.entry_rows < a.M ? m0 + pack * a.entry_rows : a.M;
  } else if (kTiling == kTilingEntries && a.entry_rows > 0) {
    const int64_t tm = (a.entry_rows + TM - 1) / TM;
    const int64_t e = t / (tm * tn), r = t - e * (tm * tn);
    const int64_t i = r / tn;
    m0 = e * a.entry_rows + i * TM;
    n0 = (r - i * tn) * TN;
    nb0 = (a.entry0 + e) * a.N + n0;
    m_end = (e + 1) * a.entry_rows;
  } else {
    if (kTiling == kTilingListed) t = a.tile_list[1 + t];
    m0 = (t / tn) * TM;
    n0 = (t - (t / tn) * tn) * TN;
    nb0 = n0;
    m_end = a.M;
  }
}
// Moduli a GEMM launch computes (every CTA reads the same device int).
// A count of 0 means the launch has nothing to compute (no work item).
__device__ __forceinline__ int planes_used(const ResGemmArgs& a) {
  if (a.used == nullptr) return a.nplanes;
  const int u = *a.used;
  if (u <= 0) return 0;
  return u < a.used_min ? a.used_min : (u > a.nplanes ? a.nplanes : u);
}
// The same GEMM with 256 x 256 tiles over CTA pairs (cta_group::2); returns
// cudaErrorNotSupported (nothing enqueued) where clusters of two cannot run.
cudaError_t launch_residue_gemm_pair(const ResGemmArgs& a, cudaStream_t stream);

}  // namespace det
