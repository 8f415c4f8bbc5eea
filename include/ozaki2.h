/*
 * ozaki2.h — C ABI of the GB300 (sm_103a) Ozaki Scheme II FP64 GEMM.
 *
 * The library computes C = A B for FP64 matrices through s small integer
 * channels, following the pipeline of "Profiling Ozaki II: The Cost Behind
 * Fast INT8 GEMMs" (§1, pipeline table) and "Ozaki II supplement: INT8 range
 * conditions and paper performance results" (§1.1):
 *
 *   1. choose power-of-two row scales D = diag(2^alpha_i) and column scales
 *      E = diag(2^beta_j) from a bound on |A||B| (fast: Cauchy–Schwarz norm
 *      bound; accu: one extra integer bound GEMM — "Profiling Ozaki II" §2),
 *   2. A' = trunc(D A), B' = trunc(B E), then the centered residues
 *      A_t = rho_{m_t}(A'), B_t = rho_{m_t}(B') for s pairwise-coprime
 *      moduli m_t <= 256 (supplement §1.2),
 *   3. P_t = A_t B_t exactly, R_t = P_t mod m_t in [0, m_t),
 *   4. X = CRT_M(R_1..R_s) in [-M/2, M/2), C = D^-1 X E^-1.
 *
 * Moduli: the s largest integers <= 256 taken greedily, each coprime to all
 * larger ones kept (256, 255, 253, 251, 247, 241, 239, 233, ...).
 *
 * Layouts: every matrix is column-major.  A is p x q with leading dimension
 * lda >= p, B is q x r (ldb >= q), C is p x r (ldc >= p).  C is overwritten
 * (there are no BLAS alpha/beta scalars).  A, B and C are caller-owned device
 * memory (ozaki2_dgemm_host excepted) and C must not overlap A or B.
 *
 * Asynchrony: ozaki2_dgemm is ordered after earlier work on `stream` (a
 * cudaStream_t; NULL means the legacy default stream), later work on
 * `stream` is ordered after it, and it returns without synchronising.
 * Inside, the overlapped schedule also runs kernels on two library-owned
 * streams of the same workspace, joined to `stream` by events: a second
 * stream for preprocessing and the CRT, and a stream at the device's
 * greatest priority for the GEMMs.  Argument errors are returned before
 * anything is enqueued.
 *
 * Workspace: intermediate planes, residues and exponents live in a
 * library-owned device workspace, one per (device, stream) pair, grown on
 * demand and kept for later calls.  Growing it synchronises the device.
 * Calls on the same stream are ordered; calls that share a stream's
 * workspace must not run concurrently from several host threads.
 *
 * Preconditions: finite inputs (an Inf/NaN entry gives an unspecified
 * result in its row of C / column of C), 2 <= s <= 20, and the inner
 * dimension within its mode's limit below.  The INT32 condition q < 131072
 * of "Ozaki II supplement: INT8 range conditions and paper performance
 * results" §1.3 bounds one unblocked accumulation; the modular GEMMs here
 * reduce every K-block of at most 960 terms (1024 for odd m_t) modulo m_t before the next is
 * added (the blocking that section describes for larger q), so the result
 * R_t = P_t mod m_t is exact for any q.  What remains: the fast-mode
 * sum-of-squares statistic is a 64-bit sum of q terms below 2^40
 * (q < 2^24); the accu bound product Wbar = Abar Bbar is accumulated
 * exactly in INT32 (q 127^2 < 2^31, q <= 133144); the checking output P of
 * ozaki2_dgemm_debug is int32 (q < 131072).
 */
#ifndef OZAKI2_H
#define OZAKI2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OZ2_FAST = 0, /* row/column norm bound (Cauchy–Schwarz) */
  OZ2_ACCU = 1  /* one extra bound GEMM on upward-quantised |A|, |B| */
} oz2_mode;

typedef enum {
  OZ2_OK = 0,
  OZ2_ERR_INVALID_ARG = 1,       /* bad size, leading dimension, pointer, s or mode */
  OZ2_ERR_Q_TOO_LARGE = 2,       /* q at or above its mode's limit (OZ2_Q_LIMIT_*) */
  OZ2_ERR_NO_MEMORY = 3,         /* workspace allocation failed */
  OZ2_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
  OZ2_ERR_DEVICE_TIMEOUT = 5,    /* a bounded device-side wait gave up */
  OZ2_ERR_UNSUPPORTED_DEVICE = 6, /* the current device is not sm_103 */
  OZ2_ERR_SCRATCH_TOO_SMALL = 7   /* p + r exceeds OZ2_NOALLOC_MAX_VECTORS */
} oz2_status;

/* Smallest and largest number of moduli accepted. */
#define OZ2_S_MIN 2
#define OZ2_S_MAX 20
/* Exclusive upper bounds on the inner dimension q (see the file comment). */
#define OZ2_Q_LIMIT_FAST (1 << 24)   /* fast mode */
#define OZ2_Q_LIMIT_ACCU 133145      /* accu mode: q 127^2 < 2^31 */
#define OZ2_Q_LIMIT_P 131072         /* ozaki2_dgemm_debug with P requested: q 2^14 < 2^31 */

/*
 * C = A B by Ozaki Scheme II with s moduli and the given bound mode.
 * A, B, C: device pointers.  stream: cudaStream_t (may be NULL).
 * Returns OZ2_OK once every kernel is enqueued; see the file comment for
 * the errors returned synchronously.
 */
oz2_status ozaki2_dgemm(int64_t p, int64_t q, int64_t r,
                        const double* A, int64_t lda,
                        const double* B, int64_t ldb,
                        double* C, int64_t ldc,
                        int s, oz2_mode mode, void* stream);

/*
 * The same pipeline, run by the same kernels, with each stage's output
 * copied out for checking.  Every output pointer may be NULL (skipped).
 * All are device pointers, owned by the caller:
 *   alpha [p] int32, beta [r] int32   — the exponents of D and E;
 *   Ares  [s][p][q] int8              — rho_{m_t}(A'), row-major per plane;
 *   Bres  [s][r][q] int8              — rho_{m_t}(B'), column j contiguous;
 *   P     [s][r][p] int32             — A_t B_t, column-major per plane
 *                                       (computed by an extra GEMM launch
 *                                       that keeps exact sums);
 *   R     [s][r][p] uint8             — P_t mod m_t, column-major per plane;
 *   X     [r][p][3] uint64            — CRT integer, 192-bit two's
 *                                       complement, little-endian limbs,
 *                                       column-major over (i, j).
 * The call synchronises `stream` before returning.
 */
oz2_status ozaki2_dgemm_debug(int64_t p, int64_t q, int64_t r,
                              const double* A, int64_t lda,
                              const double* B, int64_t ldb,
                              double* C, int64_t ldc,
                              int s, oz2_mode mode, void* stream,
                              int32_t* alpha, int32_t* beta,
                              int8_t* Ares, int8_t* Bres,
                              int32_t* P, uint8_t* R, uint64_t* X);

/*
 * ozaki2_dgemm with CUDA events recorded between its stages; synchronises
 * `stream` and writes the milliseconds of each stage to stage_ms[0..5]:
 *   0 scale statistics and exponents (fast) or bound quantisation (accu);
 *     in fast mode with q <= 8192 also B's residue planes, made together
 *     with B's statistics (one kernel reading B once up to q = 2048; above
 *     that a statistics kernel, then the residue kernel)
 *   1 bound GEMM and exponents (accu; 0 in fast mode)
 *   2 residue planes of A and (unless made in stage 0) of B
 *   3 the s modular GEMMs with the fused mod-m_t epilogue
 *   4 CRT and inverse scaling
 *   5 the whole call
 */
oz2_status ozaki2_dgemm_stages(int64_t p, int64_t q, int64_t r,
                               const double* A, int64_t lda,
                               const double* B, int64_t ldb,
                               double* C, int64_t ldc,
                               int s, oz2_mode mode, void* stream, float* stage_ms);

/*
 * Host-memory variant: A, B and C are HOST pointers (pinned memory gives the
 * fastest copies).  The library copies A and B into a device staging area of
 * its workspace, runs ozaki2_dgemm on `stream`, copies C back, and
 * synchronises `stream` before returning.  With the overlapped schedule the
 * copies are part of it: A's row blocks and B's column parts go up on a
 * library-owned stream in the order the kernels consume them, and each part
 * of C comes back as soon as its CRT has finished.
 */
oz2_status ozaki2_dgemm_host(int64_t p, int64_t q, int64_t r,
                             const double* A, int64_t lda,
                             const double* B, int64_t ldb,
                             double* C, int64_t ldc,
                             int s, oz2_mode mode, void* stream);

/*
 * Stage profiling.  After ozaki2_profile_begin(max_calls), each of the next
 * max_calls ozaki2_dgemm calls records CUDA events at its stage boundaries
 * without synchronising.  ozaki2_dgemm overlaps stages (row blocks: the
 * statistics and residues of block b+1 and the CRT of block b run on a second
 * stream while the GEMMs of block b run on the library's GEMM stream), so
 * here stage 0 covers the statistics of A's first row block (with all of B's
 * side running beside it on the second stream), stage 2 is the residue time
 * before the first GEMM starts, stage 3 the span of all GEMM launches, and
 * stage 4 the CRT time after the last GEMM; stages 0, 1 and 5
 * are as for ozaki2_dgemm_stages, which runs the stages one after another.
 * ozaki2_profile_end synchronises those events, writes the per-stage
 * milliseconds summed over the recorded calls to stage_ms_sum[0..5] and the
 * number of recorded calls to *ncalls, and turns recording off.
 */
oz2_status ozaki2_profile_begin(int max_calls);
oz2_status ozaki2_profile_end(float* stage_ms_sum, int* ncalls);

/* Number of kernels this library has launched so far in this process. */
uint64_t ozaki2_launch_count(void);

/* Largest p + r that ozaki2_fast_exponents_noalloc accepts (16 MiB of scratch). */
#define OZ2_NOALLOC_MAX_VECTORS (1 << 20)

/*
 * Fast-mode exponents without any device allocation.  The paper has no
 * counterpart: this entry point exists for callers that must not allocate
 * device memory themselves or through the library, such as frameworks that
 * hand out all device memory from their own pool, latency-critical loops
 * where cudaMalloc could block or synchronise, and plug-ins that are not
 * allowed to use the allocator.
 *
 * Computes alpha[p] and beta[r], the row and column exponents that
 * ozaki2_dgemm uses in OZ2_FAST mode for the same A, B and s (see
 * ozaki2_dgemm_debug), enqueued on `stream`.  A, B, alpha and beta are
 * caller-owned device memory, layouts as for ozaki2_dgemm.
 *
 * Scratch: a fixed array of 2 * OZ2_NOALLOC_MAX_VECTORS 64-bit words inside
 * the library, resident on every device that loads the library until the
 * process exits.  Calls with p + r > OZ2_NOALLOC_MAX_VECTORS return
 * OZ2_ERR_SCRATCH_TOO_SMALL before enqueuing anything.  Every call shares
 * that array and clears the part it uses; calls whose kernels overlap on the
 * GPU (e.g. on unordered streams) race on it and give wrong exponents.
 *
 * The first call on each device looks up the array's device address (this
 * may load the library's device code on that device); make that first call
 * before any stream capture.  No call allocates device memory.
 */
oz2_status ozaki2_fast_exponents_noalloc(int64_t p, int64_t q, int64_t r,
                                         const double* A, int64_t lda,
                                         const double* B, int64_t ldb,
                                         int s, int32_t* alpha, int32_t* beta,
                                         void* stream);

/* Writes the s moduli to out[0..s-1]; returns s, or -1 if s is out of range. */
int ozaki2_moduli(int s, int32_t* out);

/*
 * Sticky device-side error word: OZ2_ERR_DEVICE_TIMEOUT if a bounded wait in
 * any kernel that has completed gave up since the last call, else OZ2_OK.
 * Reading it clears it.  Synchronise the stream first to include its work.
 */
oz2_status ozaki2_last_error(void);

/* Frees every workspace of every device (synchronises each device first). */
void ozaki2_workspace_release(void);

/* Static text for a status code. */
const char* ozaki2_status_string(oz2_status status);

/*
 * Self-test of the bounded-wait machinery: launches one block that waits on
 * a barrier nothing completes, with a wait limit of about `limit_us`
 * microseconds (1..1000000).  It returns OZ2_ERR_DEVICE_TIMEOUT when the
 * wait gave up as designed and the kernel exited cleanly, OZ2_OK if it did
 * not (a bug), or OZ2_ERR_CUDA.  Synchronises the device.
 */
oz2_status ozaki2_selftest_wait_timeout(int limit_us);

#ifdef __cplusplus
}
#endif

#endif /* OZAKI2_H */
