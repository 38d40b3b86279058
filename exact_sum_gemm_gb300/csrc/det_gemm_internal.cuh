// Shared constants and launch plumbing of the exact GEMM kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "det_kernels.h"

namespace det {

constexpr int kTile = 64;                 // band kernel output tile (and routing unit)
constexpr int kDeepGap = 18;              // "deep" element: more than 18 binades below its row max
constexpr int kEmaxEmpty = static_cast<int>(0x80808080u);   // memset(0x80) pattern: no live element

// Device scratch of one det_gemm / det_gemm_partial call.
struct Scratch {
  int* emaxA;          // [M]   (emaxB follows contiguously)
  int* emaxB;          // [N]
  int* deepA;          // [M]   (deepB follows contiguously)
  int* deepB;          // [N]
  uint8_t* route;      // [tiles of 64x64]: 1 = general kernel
  int* general;        // [1 + tiles]: count, then the indices of the tiles routed to the general kernel
  int* bmax;           // [tiles_m + tiles_n]: largest deep count per 64-row / 64-column block
  int64_t* fallback;   // [slots][kPlanes][kTile*kTile] band-kernel fallback digits (det_gemm only)
  int64_t slots;       // resident band-kernel CTAs (fallback regions)
};

// Bytes of scratch a call needs, and how to carve it out of one allocation.
size_t scratch_bytes(const GemmArgs& g, int64_t slots);
Scratch carve_scratch(void* base, const GemmArgs& g, int64_t slots);

// Capacity of a row's deep-element list; a 64x64 tile whose worst row plus
// worst column hold more deep elements goes to the general kernel.
int deep_list_cap(int64_t K);
cudaError_t launch_prepass(const GemmArgs& g, const Scratch& s, cudaStream_t stream);
// The residue path's pieces of the pre-pass: row maxima only, and routing from
// deep counts produced elsewhere (the residue kernel's list counters).
cudaError_t launch_emax(const GemmArgs& g, const Scratch& s, cudaStream_t stream);
// Routing from deep counts; with deep_rows [M] / deep_cols [N] /
// deep_counters (two ints, zero at launch) it also lists the rows and columns
// holding deep elements (residue path), else pass null.
cudaError_t launch_classify(const GemmArgs& g, const int* deepA, const int* deepB, const Scratch& s,
                            int* deep_rows, int* deep_cols, int* deep_counters,
                            cudaStream_t stream);
cudaError_t launch_band(const GemmArgs& g, const Scratch& s, cudaStream_t stream);
// General kernel over the 64x64 tiles listed in general (count first).
// allow_split: when the grid would hold few tiles and K is long, K may be
// split among CTAs with a scratch slot per tile from the library's pool
// (false: allocate nothing).
cudaError_t launch_kulisch(const GemmArgs& g, const int* general, bool allow_split,
                           cudaStream_t stream);

// The general tiles of a residue-path call (route and list in s): the wide
// residue path where the tiles' rows span at most its window and are finite,
// the general kernel for the rest.  wide_prepare: statistics, norms and
// planes on `stream`, then ev_planes; wide_finish: the wide tensor-core GEMM,
// its reconstruction and the general kernel on `tail`, after ev_planes.
struct WidePlan {
  bool active;                // false: the problem is too large, general kernel only
  const int* general;         // the narrow routing's list of general tiles
  void* mem;                  // scratch, released on the tail stream
  int* wide;                  // wide tiles (count first)
  int* rest;                  // tiles left for the general kernel (count first)
  int* glist;                 // the wide GEMM's output tiles holding a wide tile (count first)
  void* ctl;                  // moduli count, error flag, counters
  __nv_bfloat16* planesA;
  __nv_bfloat16* planesB;
  int8_t* res;
  const int* loA;             // exponent keys of the rows' smallest elements
  const int* loB;
  int pmax;
  int64_t Kp;
};
cudaError_t wide_prepare(const GemmArgs& g, const Scratch& s, cudaStream_t stream,
                         cudaEvent_t ev_planes, WidePlan* plan);
cudaError_t wide_finish(const GemmArgs& g, const WidePlan& plan, cudaStream_t tail,
                        cudaEvent_t ev_planes);
// Diagnostic: the last residue-path call's 64x64 tiles (all, general before
// the wide split, wide, left for the general kernel); synchronises.
int route_record(long long* out);

// Pre-pass + band + general kernels with caller-provided scratch of at least
// scratch_bytes(g, slots) bytes (256-byte aligned); allow_alloc lets the
// general kernel take a K-split slot from the library's pool.
cudaError_t run_gemm_with_scratch(const GemmArgs& g, void* scratch, int64_t slots,
                                  bool allow_alloc, cudaStream_t stream);

// det_gemm_partial_noalloc: scratch from a fixed static device array.
bool noalloc_fits(const GemmArgs& g);
cudaError_t launch_gemm_partial_noalloc(const GemmArgs& g, cudaStream_t stream);

// Band-kernel CTAs resident on the current device (persistent grid size).
int64_t band_slots(const GemmArgs& g);

}  // namespace det
