/*
 * det_gemm.h -- C ABI of the exact-sum (Kulisch long-accumulator) GEMM.
 *
 * What the library computes (det-train page, section "Method"): every output
 * of C = A * B^T is the exact sum of its bf16/f32 products, kept as signed
 * int64 digits of radix 2^32 wide enough for any fp32 x fp32 product, then
 * carry-normalised and rounded to fp32 exactly once, to nearest with ties to
 * even.  Integer addition is associative, so the result does not depend on
 * tiling, K-sharding, fold order or repetition, and digit arrays of K-shards
 * combine by plain addition.
 * The call names follow the page's usage section: det_gemm, det_gemm_partial,
 * det_combine, det_finalize, and the forward/dgrad/wgrad of DetLinear.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All data pointers are DEVICE pointers (CUDA), owned by the caller.  The
 *    library never frees or retains them, and never synchronises the stream:
 *    every call only enqueues work on `stream` (a cudaStream_t; NULL means the
 *    legacy default stream) and returns.
 *  - Operands: A is logically [M, K] and B is logically [N, K] ("x" and "w" of
 *    the page, w laid out like nn.Linear.weight).  op = 0: the operand is
 *    stored row-major as [rows, K] with K contiguous, element (r, k) at
 *    X[r * ld + k], ld >= K.  op = 1: it is stored as [K, rows] with rows
 *    contiguous, element (r, k) at X[k * ld + r], ld >= rows.
 *    Both operands have the same dtype (DET_F32 or DET_BF16 bit patterns).
 *  - Output C is fp32 [M, N] row-major, element (m, n) at C[m * ldc + n].
 *  - K <= DET_K_MAX per call (det-train page, "Requirements and limits").
 *    K = 0 is allowed: every digit is zero and every output is +0.0f.
 *  - Digit arrays ("partials") are int64, planar [DET_PLANES][M][N],
 *    contiguous: planes 0..17 are the digits (digit j weighs 2^(32j-298);
 *    the smallest nonzero |product| is 2^-298 and the largest is below
 *    2^256), plane 18 counts the products summed, plane 19 counts products
 *    with a non-finite operand.  Arrays written by this library are canonical:
 *    digits 0..16 in [0, 2^32), digit 17 signed.
 *  - Rounding: exact zero -> +0.0f; a nonzero sum that rounds to zero keeps
 *    its sign; overflow -> +-inf; an output with any non-finite product is the
 *    canonical NaN 0x7FC00000 (the page does not treat Inf/NaN inputs).
 *  - Errors: argument errors are detected on the host and returned before
 *    anything is enqueued.  DET_ERR_CUDA reports a failed launch or CUDA call;
 *    nothing throws across the ABI.
 */
#ifndef DET_GEMM_H
#define DET_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DET_OK = 0,
  DET_ERR_INVALID_ARG = 1, /* null pointer, bad op flag or leading dimension */
  DET_ERR_DTYPE = 2,       /* dtype is not DET_F32 / DET_BF16 */
  DET_ERR_SHAPE = 3,       /* negative or too large M, N, K or part count */
  DET_ERR_K_LIMIT = 4,     /* K > DET_K_MAX */
  DET_ERR_OVERFLOW = 5,    /* digit headroom would be exceeded (combine of too many parts) */
  DET_ERR_ALIGNMENT = 6,   /* a pointer is not aligned to its element size */
  DET_ERR_CUDA = 7,        /* a CUDA call or kernel launch failed */
  DET_ERR_NOALLOC_LIMIT = 8, /* problem too large for det_gemm_partial_noalloc's fixed scratch */
  DET_ERR_TIMEOUT = 9        /* a bounded wait inside a kernel ran out (det_device_status) */
} det_status;

typedef enum { DET_F32 = 0, DET_BF16 = 1 } det_dtype;

enum {
  DET_DIGITS = 18,             /* radix-2^32 digits per output */
  DET_PLANES = 20,             /* digits + product count + non-finite count */
  DET_K_MAX = 1 << 19,         /* largest K of one GEMM call */
  DET_MAX_COMBINE = 1 << 20    /* most partials one det_combine call accepts */
};

/* Version of this ABI (bumped on any incompatible change). */
int det_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* det_status_string(det_status s);

/* Number of kernels this library has enqueued in this process so far (all
 * devices, all threads).  A diagnostic for benchmarks and tests. */
uint64_t det_kernel_launches(void);

/* Per-stage device timing, a diagnostic for benchmarks.  det_stage_timing(1)
 * brackets every stage of the following det_gemm / det_gemm_partial calls
 * (exponent pre-pass, residue planes, residue GEMM on the tensor cores,
 * reconstruction, general kernel, band kernel) with CUDA events recorded on
 * the call's stream; det_stage_timing(0) stops.  Returns the previous
 * setting.  After the caller has synchronised those streams,
 * det_stage_report writes up to `max` entries (stage name -- a static string
 * --, total milliseconds, number of timed launches), clears the record and
 * returns the number of entries.  Any output pointer may be NULL. */
int det_stage_timing(int enable);
int det_stage_report(const char** names, double* total_ms, int* counts, int max);

/* The same records as a timeline, in the order the stages were enqueued:
 * stage name, start and stop in milliseconds from the first record's start.
 * Tensor-core launches ("residue_gemm") sit on two library streams and
 * overlap the stages on the call's stream (and, at a band change, one
 * another); a record starts when its stream reaches it, which may precede
 * its first kernel's start.  Writes up to `max`
 * entries, clears the record and returns the number written.  Any output
 * pointer may be NULL. */
int det_stage_timeline(const char** names, double* start_ms, double* stop_ms, int max);

/* Device-side status of the library on the current device.  The tensor-core
 * kernels bound every wait on a barrier (about 2 s); if one runs out, that
 * call's outputs are the canonical NaN and the kernel records the expiry in a
 * per-device word, which stays set until cleared.  det_device_status returns
 * DET_ERR_TIMEOUT if it is set, DET_OK if not (DET_ERR_CUDA if it cannot be
 * read), and resets it when `clear` is nonzero.  It synchronises the device
 * first, so it sees every call enqueued before it.  A diagnostic, not part of
 * the page's calls. */
det_status det_device_status(int clear);

/* Self-test of that mechanism: enqueues on `stream` one small kernel that
 * waits, with the same bounded-wait routine as the tensor-core kernels, on a
 * barrier that nothing ever releases; after limit_ns nanoseconds (1 ..
 * 10^9, else DET_ERR_INVALID_ARG) the wait gives up, records the expiry in the
 * status word as those kernels do, and the kernel returns.  No memory is
 * written but that word; the device stays usable. */
det_status det_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Scratch memory.  det_gemm and det_gemm_partial (and the bias variants)
 * take their working memory per call, stream-ordered, from a memory pool that
 * the library creates per device; it is released on the call's stream when
 * the call's work is done.  By default the pool keeps the freed memory
 * reserved for the next call (a 4096^3 f32 det_gemm uses about 1.1 GB), so
 * repeated calls do not go back to the driver.
 *   det_release_scratch: synchronises the current device, then returns all
 *     of its pool's unused memory to the device.
 *   det_set_scratch_retention: bytes each pool keeps reserved after its
 *     memory is freed; 0 returns freed scratch at the next synchronisation
 *     (slower repeated calls), UINT64_MAX (the default) keeps it all.
 *   det_scratch_stats: allocations the library has taken from its pools so
 *     far (all devices), and the current device's reserved and in-use pool
 *     bytes (0 before its first allocation).  Any pointer may be NULL.
 * Stream use: besides the caller's stream, the residue path runs on five
 * library streams per device (two of the greatest priority for the
 * tensor-core launches, and three for overlapped reconstruction and general
 * tiles), joined back to the caller's stream by events before the call
 * returns.  Calls from different caller streams on one device share those
 * streams, so their tensor-core work runs one call after the other; the
 * enqueue itself is serialised by a lock. */
det_status det_release_scratch(void);
det_status det_set_scratch_retention(uint64_t bytes);
det_status det_scratch_stats(uint64_t* allocations, uint64_t* reserved_bytes,
                             uint64_t* used_bytes);

/* Pipe-throughput microbenchmark (a diagnostic: the roofline denominators of
 * exact accumulation on the CUDA cores; the page's kernel runs on the fp64
 * scalar cores, section "Measured").  Enqueues on `stream` one launch of
 * `blocks` blocks of det_pipe_benchmark_threads_per_block() threads; each
 * thread performs iters * det_pipe_benchmark_ops_per_thread_iter()
 * operations of one kind, each a single instruction in a dependency ring of
 * independent accumulators, and writes one 32-bit word to out[thread] (a
 * device buffer of blocks * threads words, so the work cannot be dropped).
 * The caller times the launch (CUDA events) and divides the operation count
 * by the time.  iters >= 1, 1 <= blocks <= 2^20. */
enum {
  DET_PIPE_IADD = 0,        /* 32-bit integer add (add.u32) */
  DET_PIPE_LOP3 = 1,        /* three-input logic op (lop3.b32) */
  DET_PIPE_IMAD = 2,        /* 32-bit integer multiply-add, low half (mad.lo.u32) */
  DET_PIPE_IMAD_WIDE = 3,   /* 32 x 32 -> 64-bit multiply-add (mad.wide.u32) */
  DET_PIPE_FFMA = 4,        /* fp32 fused multiply-add */
  DET_PIPE_DFMA = 5         /* fp64 fused multiply-add */
};
det_status det_pipe_benchmark(int kind, int64_t iters, int64_t blocks, void* out, void* stream);
int det_pipe_benchmark_ops_per_thread_iter(void);
int det_pipe_benchmark_threads_per_block(void);

/* The wide residue path (see det_tile_routes) on (enable != 0, the default)
 * or off for the following calls from any thread; returns the previous
 * setting.  Results are identical either way (every path computes the same
 * exact sum); with the path off, tiles the narrow residue path leaves go to
 * the general kernel on the CUDA cores, and a call enqueues about eight fewer
 * kernels, which callers whose data is known to span few binades may prefer. */
int det_set_wide_path(int enable);

/* Strided batches (det_gemm_strided_batched) as one pipeline where their
 * shapes allow (1, the default) or entry by entry (0); returns the previous
 * setting.  The results are the same bytes; the switch exists so that the
 * two can be timed against each other. */
int det_set_batched_pipeline(int enable);

/* Diagnostic for tests and benchmarks: how the most recent residue-path
 * det_gemm / det_gemm_partial call on the current device routed its 64x64
 * output tiles.  out[0] = all tiles, out[1] = tiles the narrow residue path
 * left ("general": more elements more than 18 binades below their row's
 * largest than its lists take), out[2] = of those, tiles the wide residue
 * path computed (every row of A and of B in the tile finite and spanning at
 * most 88 binades for f32, 124 for bf16), out[3] = tiles left for the general
 * Kulisch kernel.  Returns 0, or -1 (null out, CUDA error).  Reads device
 * memory, so it synchronises with the device; calls that take the band path
 * (K = 0, very large grids) do not update it. */
int det_tile_routes(int64_t* out);

/* Worst-case number of moduli (bf16 tensor-core GEMMs) of det_gemm's residue
 * path for this dtype and K: enough that their product exceeds twice the
 * largest possible |sum of shallow products|.  The residue planes are written
 * for this many; a row band may compute fewer (det_moduli_used).  0 for
 * K = 0; -1 for bad arguments. */
int det_residue_moduli(det_dtype dtype, int64_t K);

/* Diagnostic for benchmarks: the moduli counts the most recent residue-path
 * det_gemm / det_gemm_partial call on the current device used, one per row
 * band of C, in band order.  The planes are written for det_residue_moduli's
 * worst-case count; each band then computes only as many moduli as a
 * Cauchy-Schwarz bound of its exact dot products needs (|S| <= |row of A|
 * |row of B| on the integer grid; fewer moduli for typical data).  Writes up
 * to `max` counts to `out` (may be NULL) and returns how many the call had
 * (capped at `max`), or -1 on a CUDA error.  Reads device memory, so it
 * synchronises with the device; concurrent calls overwrite one another's
 * record. */
int det_moduli_used(int* out, int max);

/*
 * det_gemm -- C = RNE_f32( sum_k A(m,k) * B(n,k) ), computed exactly.
 * det-train page, usage section (the det_gemm call) and section "Method".
 * Enqueues the exponent pre-pass and the accumulate kernel on `stream`; the
 * digits are never written to memory (finalize is fused).  A and B must be
 * aligned to their element size, C to 4 bytes.
 */
det_status det_gemm(det_dtype dtype, int64_t M, int64_t N, int64_t K,
                    const void* A, int64_t lda, int opA,
                    const void* B, int64_t ldb, int opB,
                    float* C, int64_t ldc, void* stream);

/*
 * det_gemm_partial -- the same exact accumulation, written out unrounded as a
 * canonical digit array P [DET_PLANES][M][N] (8-byte aligned, contiguous,
 * M*N*160 bytes).  det-train page, usage section (the det_gemm_partial
 * call) and section "Method" (partials of K-shards add up to the full sum).
 * Plane 18 is set to K.
 */
det_status det_gemm_partial(det_dtype dtype, int64_t M, int64_t N, int64_t K,
                            const void* A, int64_t lda, int opA,
                            const void* B, int64_t ldb, int opB,
                            int64_t* P, void* stream);

/*
 * det_combine -- out = sum_i parts[i], elementwise over all DET_PLANES planes,
 * then carry-normalised to canonical form.  det-train page, usage section
 * (the det_combine call) and section "Method".  `parts` is a HOST array of
 * n >= 1 device pointers, each to a [DET_PLANES][M][N] int64 array; `out` may
 * alias any of them.  Inputs need not be canonical, but the per-digit sums
 * must stay below 2^62 in magnitude (always true for up to DET_MAX_COMBINE
 * canonical parts).  n > DET_MAX_COMBINE returns DET_ERR_OVERFLOW.
 */
det_status det_combine(int64_t M, int64_t N, const int64_t* const* parts, int n,
                       int64_t* out, void* stream);

/*
 * det_finalize -- round a digit array once to fp32.  det-train page, usage
 * section (the det_finalize call) and section "Method" (carry-normalise, round
 * once, round-to-nearest-even).  P is [DET_PLANES][M][N] int64 with digits of
 * magnitude below 2^62; C is fp32 [M, N] with leading dimension ldc >= N.
 */
det_status det_finalize(int64_t M, int64_t N, const int64_t* P, float* C, int64_t ldc,
                        void* stream);

/*
 * det_gemm_partial_noalloc -- det_gemm_partial that allocates no memory.
 * The det-train page has no counterpart: this entry point exists for callers
 * that cannot call cudaMalloc -- for example a plug-in inside a host framework
 * that owns all device memory and forbids allocations behind its back, or
 * latency-critical code that must not enter the CUDA allocator (which may
 * synchronise the device).  Arguments, output and result are exactly those of
 * det_gemm_partial; the caller still provides A, B and P.
 *
 * The working memory (per-row exponent maxima, deep-element counts and the
 * tile routing table) lives in one fixed array of DET_NOALLOC_SCRATCH_BYTES
 * bytes that is a static device variable of this library: every GPU that
 * loads the library holds it until the process exits.  With Tm = ceil(M/64),
 * Tn = ceil(N/64), T = Tm * Tn and a(x) = x rounded up to a multiple of 256,
 * a call needs
 *     2 a(4 (M + N)) + a(T) + a(4 (T + 1)) + a(4 (Tm + Tn))   bytes
 * (exponent maxima and deep counts of every row and column; one routing byte
 * and one list entry per 64x64 output tile; the largest deep count per
 * 64-row and 64-column block).  M = N = 20000 fits (812,544 bytes); M = N =
 * 24576 does not (1,133,824); with M = 1, N may reach 128,767.  Larger
 * problems return DET_ERR_NOALLOC_LIMIT before anything is enqueued.
 *
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * Every call uses the same array and clears what must start at zero; two calls
 * whose work overlaps on the GPU (e.g. on different streams without ordering)
 * race on it and give undefined results.
 */
enum { DET_NOALLOC_SCRATCH_BYTES = 1 << 20 };
det_status det_gemm_partial_noalloc(det_dtype dtype, int64_t M, int64_t N, int64_t K,
                                    const void* A, int64_t lda, int opA,
                                    const void* B, int64_t ldb, int opB,
                                    int64_t* P, void* stream);

/*
 * DetLinear (det-train page, usage section: a 4096 -> 4096 layer whose
 * forward and backward passes are both deterministic).
 * Bias-free; every GEMM is an exact det_gemm:
 *   forward: y[b,o]  = sum_i x[b,i]  W[o,i]   x [batch,in], W [out,in], y [batch,out]
 *   dgrad:   dx[b,i] = sum_o dy[b,o] W[o,i]   dy [batch,out], dx [batch,in]
 *   wgrad:   dW[o,i] = sum_b dy[b,o] x[b,i]   dW [out,in]  (K = batch <= DET_K_MAX)
 * All tensors are contiguous row-major; gradients are fp32.
 */
det_status det_linear_forward(det_dtype dtype, int64_t batch, int64_t in_features,
                              int64_t out_features, const void* x, const void* W, float* y,
                              void* stream);
det_status det_linear_dgrad(int64_t batch, int64_t in_features, int64_t out_features,
                            const float* dy, const float* W, float* dx, void* stream);
det_status det_linear_wgrad(int64_t batch, int64_t in_features, int64_t out_features,
                            const float* dy, const float* x, float* dW, void* stream);

/*
 * det_linear_forward_bias -- y[b,o] = RNE_f32( sum_i x[b,i] W[o,i] + bias[o] ),
 * the bias being one more exact term of the same sum, rounded with it once.
 * The det-train page shows a bias-free layer; this is its bias-carrying form:
 * the product 1 * bias[o] joins the exact accumulation, so the result keeps
 * every invariance of det_gemm.  bias [out] is contiguous and has the dtype
 * of x and W (a null bias is det_linear_forward).  Needs in + 1 <= DET_K_MAX.
 * Scratch: (batch + out) * (in + 1) elements from the library's memory pool
 * for the widened operands [x | 1] and [W | bias], released on `stream`.
 */
det_status det_linear_forward_bias(det_dtype dtype, int64_t batch, int64_t in_features,
                                   int64_t out_features, const void* x, const void* W,
                                   const void* bias, float* y, void* stream);

/*
 * det_linear_bias_grad -- db[o] = RNE_f32( sum_b dy[b,o] ), exact (the
 * gradient of the bias term above).  dy fp32 [batch, out] contiguous, db fp32
 * [out]; batch <= DET_K_MAX.  Scratch: batch floats from the memory pool.
 */
det_status det_linear_bias_grad(int64_t batch, int64_t out_features, const float* dy, float* db,
                                void* stream);

/*
 * det_gemm_strided_batched -- `batch` independent exact GEMMs,
 *   C_b = RNE_f32( A_b * B_b^T ),  b = 0 .. batch-1,
 * with A_b = A + b * strideA, B_b = B + b * strideB (in elements of the
 * operand dtype) and C_b = C + b * strideC (floats); every matrix uses the
 * layout rules of det_gemm (lda/opA, ldb/opB, ldc).  A stride of 0 shares
 * one operand across the batch.  The det-train page has no batched call; it
 * names reproducible training under sequence parallelism among its
 * references (section "References"), whose per-head attention products are
 * batches of small independent GEMMs.  Each C_b is bitwise the det_gemm of
 * its operands.  The C_b must not overlap.  Negative strides return
 * DET_ERR_SHAPE.
 *
 * Where M and N are multiples of 64 and both operands are K-contiguous
 * (opA = opB = 0) with rows the fused residue kernel reads by vector loads
 * (K <= 4096; A, B, lda, ldb, strideA and strideB 16-byte multiples for f32,
 * 8-byte for bf16), every entry runs in ONE residue-path pipeline: the
 * entries' rows are stacked, each output tile is computed from its own
 * entry's operands only, and one set of launches serves the batch (scratch
 * from the memory pool grows with batch * (M + N) rows).  Other shapes, or
 * det_set_batched_pipeline(0), enqueue the entries one after another on
 * `stream`.  Either way each C_b is bitwise the same.
 */
det_status det_gemm_strided_batched(det_dtype dtype, int64_t batch, int64_t M, int64_t N,
                                    int64_t K, const void* A, int64_t lda, int opA,
                                    int64_t strideA, const void* B, int64_t ldb, int opB,
                                    int64_t strideB, float* C, int64_t ldc, int64_t strideC,
                                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DET_GEMM_H */
