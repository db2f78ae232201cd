/*
 * bakron.h -- C ABI of libbakron.so, a GB300 (sm_103a) implementation of the
 * BaKron solver: two-sided adaptive rounding of a weight matrix under a
 * Kronecker-factored Hessian A (x) B.
 *
 * Source: "BaKron: Efficient Quantization with Kronecker-Factored Hessians"
 * (arXiv 2608.06291).
 *
 * Conventions for every entry point
 *   - Matrices are dense, row-major, 32-bit float unless stated otherwise.
 *   - W is m x n (m outputs = rows, n inputs = columns).  A (n x n) is the
 *     input-side factor and B (m x m) the output-side factor of the Hessian
 *     A (x) B of vec(W) (Sec. 3.1, Proposition 3.1: (A (x) B) vec(W) =
 *     vec(B W A^T), vec column-major).
 *   - "device" pointers must be CUDA device memory of the current device;
 *     "host" pointers are ordinary (preferably pinned) host memory.
 *   - The caller owns every buffer, including the workspace; the library
 *     allocates no memory in these calls.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream) and runs asynchronously, except where a
 *     function says it synchronizes.
 *   - Argument errors are returned synchronously before anything is
 *     enqueued.  Conditions only the device can see (a non-positive pivot,
 *     a non-finite input) are written to a caller-provided device status
 *     word; nothing traps or asserts on the device.
 *   - Return values are bakron_status codes.
 *   - Process state: the solve keeps, per device, four internal streams
 *     (tile solves and chunk products at the highest priority, mid pushes
 *     at the highest or the lowest) and a pool of ordering events (driver
 *     objects, not device memory), created
 *     by the first call on the device; the no-allocation solve caches its
 *     scratch array's device address per device.  Both caches remember the
 *     CUDA context they were made in (cuCtxGetId) and are rebuilt when the
 *     device's current context changes, e.g. after cudaDeviceReset, so the
 *     library may be used again after a reset.  Calls from several host
 *     threads on one device are serialized while they enqueue work.
 */
#ifndef BAKRON_H_
#define BAKRON_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 2: adds the row-wise, antidiagonal, alphabet, scale, packing, Hessian-factor
 * and self-test entry points; the entry points of version 1 are unchanged.
 * 3: bakron_quantize_profile reports five kernel classes (the persistent
 * sweep is class 4); adds bakron_sweep_plan_check.
 * 4: bakron_quantize runs the tile wavefront on every device (measured
 * faster than the persistent sweep on every workload); the sweep is
 * bakron_quantize_persistent, and profile class 4 stays 0.
 * 5: adds bakron_wavefront_plan_check. */
#define BAKRON_ABI_VERSION 5

typedef enum bakron_status {
  BAKRON_OK = 0,
  BAKRON_ERR_INVALID_ARG = 1, /* bad size, bit width, null pointer, aliasing */
  BAKRON_ERR_NOT_SPD = 2,     /* reserved: a factor reported a non-positive pivot */
  BAKRON_ERR_CUDA = 3,        /* a CUDA runtime call failed (launch, copy) */
  BAKRON_ERR_WORKSPACE = 4,   /* workspace null, misaligned or smaller than required */
  BAKRON_ERR_TIMEOUT = 5,     /* reserved: a bounded device-side wait gave up */
} bakron_status;

/* Device status-word bits written by bakron_quantize (0 = success). */
#define BAKRON_DEV_NONFINITE_W 1 /* W holds a NaN or an infinity */
#define BAKRON_DEV_BAD_SCALE 2   /* a scale is <= 0, NaN or infinite */
#define BAKRON_DEV_TIMEOUT 4     /* a bounded device-side wait gave up */

/* Human-readable name of a status code (static string, never NULL). */
const char* bakron_status_string(int status);

/* BAKRON_ABI_VERSION of the loaded library. */
int bakron_abi_version(void);

/* ---------------------------------------------------------------- prepare
 * Factor preparation, Sec. 3.2 Algorithm 1 prologue (also Algorithms 2, 3,
 * 5, 6; App. B: done once, at the top level):
 *     L = Cholesky(H^-1), then every column divided by its diagonal entry,
 * giving the unit lower-triangular L-hat.  Computed without forming H^-1:
 * with H = U D U^T (U unit upper triangular, factored from the last index
 * backwards), L-hat = U^-T.  Arithmetic is double-float (pairs of fp32,
 * about 44 significant bits); the result is rounded once to fp32.
 */

/* Workspace bytes bakron_factor needs for a factor of order d (d >= 1). */
size_t bakron_factor_workspace_size(int64_t d);

/* H: device, d x d, symmetric positive definite (the caller adds any
 *    damping); only the lower triangle is read.
 * Lhat: device, d x d, written in full: unit lower triangular, zeros above
 *    the diagonal.  May not alias H.
 * ws: device, >= bakron_factor_workspace_size(d) bytes, 256-byte aligned.
 * info_dev: device int32; set to 0 on success, or to 1 + the index of the
 *    first non-positive pivot met (the factorization runs from the last
 *    index backwards; Lhat is then undefined).
 */
int bakron_factor(const float* H, int64_t d, float* Lhat, void* ws, size_t ws_bytes,
                  int32_t* info_dev, void* stream);

/* Workspace bytes bakron_prepare needs (max over the two factors). */
size_t bakron_prepare_workspace_size(int64_t m, int64_t n);

/* Both factors: LA = L-hat of A (n x n), LB = L-hat of B (m x m).
 * A, B, LA, LB, ws: device.  info_dev: device int32[2], info for A then B,
 * as in bakron_factor.  The two factorizations run one after the other on
 * `stream` and share `ws`.
 */
int bakron_prepare(const float* A, const float* B, int64_t m, int64_t n, float* LA, float* LB,
                   void* ws, size_t ws_bytes, int32_t* info_dev, void* stream);

/* ---------------------------------------------------------------- quantize
 * The BaKron core, Sec. 3.5 Algorithm 6 (equal to Algorithms 2, 3, 5 by
 * Theorem 3.2): with anti-diagonals processed in order and
 *     W~ = W0 + L_B E_(earlier) L_A^T (App. B eq. (2)),
 *     v_ij = clamp(round_half_even(fp32(W~_ij) / s_i), lo, hi),
 *     E_ij = s_i v_ij - W~_ij,
 * executed as a tile wavefront: tiles on one tile anti-diagonal are solved
 * in parallel (Sec. 3.3), and the errors of a finished tile are pushed to
 * later tiles as dense products (Sec. 3.4/3.5, App. B eq. (1)).
 * All accumulation is double-float: values are unevaluated sums of two fp32
 * numbers (about 44 significant bits), products are summed with an
 * error-free offset accumulator (Rump, Ogita and Oishi, "Accurate
 * floating-point summation, part I", 2008, ExtractScalar).  The batched
 * products run on the tensor cores (tcgen05, accumulators in tensor memory)
 * through an exact split of both operands into bf16 integer digits (Ozaki,
 * Ogita, Oishi and Rump, Numer. Algorithms 2012): 5 digits per factor
 * element, 6 per double-float value, every digit-pair product and every
 * per-level sum exact in fp32.
 */

/* Workspace bytes bakron_quantize needs for an m x n problem: about 72 per
 * weight, plus, on layers of 2^22 weights and more, 10 per entry of each
 * factor (the factors' digits, computed once per solve for the chunk
 * products). */
size_t bakron_quantize_workspace_size(int64_t m, int64_t n);

/* W: device, m x n; read only.
 * LA: device, n x n unit lower-triangular L-hat of A (entries above the
 *     diagonal are ignored; the diagonal is taken as 1).
 * LB: device, m x m unit lower-triangular L-hat of B (same).
 * scales: device, m per-row scales (> 0, finite), or NULL for all ones.
 * bits: 0 for the unbounded alphabet Z (plain rounding), or 2..8 for the
 *     alphabet {-2^(bits-1) .. 2^(bits-1) - 1} (Sec. 3.1).
 * V: device int32, m x n: the integer codes.
 * Wq: device, m x n: fp32(scales[i] * V[i][j]).  W, V and Wq must be
 *     three distinct buffers.
 * ws: device, >= bakron_quantize_workspace_size(m, n) bytes, 256-byte
 *     aligned; its contents on entry do not matter.
 * status_dev: device int32; set to 0, or to an OR of BAKRON_DEV_* bits.
 *     With BAKRON_DEV_NONFINITE_W or BAKRON_DEV_BAD_SCALE set, V and Wq
 *     are undefined.
 * m, n >= 1 and m * n < 2^31.
 */
int bakron_quantize(const float* W, const float* LA, const float* LB, const float* scales, int bits,
                    int64_t m, int64_t n, int32_t* V, float* Wq, void* ws, size_t ws_bytes,
                    int32_t* status_dev, void* stream);

/* The same solve, arguments, workspace, conventions and codes (Theorem
 * 3.2: every order of the anti-diagonals that respects the dependencies
 * gives the V of App. B eq. (2)) as one persistent cooperative kernel: one
 * CTA per SM; bands of 32 rows sweep their anti-diagonals one step at a
 * time on the fp32 pipes (double-float) while the same CTAs run the
 * delayed products (Sec. 3.4/3.5) on the tensor cores from a queue of
 * tasks whose sources are complete.  CTAs wait on flags that other CTAs
 * set; every wait is bounded (about a second), and one that runs out sets
 * BAKRON_DEV_TIMEOUT in *status_dev, after which the kernel finishes
 * without waiting.  Needs cooperative launch (BAKRON_ERR_CUDA otherwise)
 * and fewer than 2^31 product tasks (BAKRON_ERR_INVALID_ARG otherwise:
 * well beyond 2^31 weights).  On a GB300 it is slower than bakron_quantize
 * on every workload measured (4096 x 4096: 22 ms against 16.7 ms): one
 * band step costs about 2 us, set by the band's write-out and by the
 * product warps sharing the SM.
 */
int bakron_quantize_persistent(const float* W, const float* LA, const float* LB, const float* scales, int bits,
                               int64_t m, int64_t n, int32_t* V, float* Wq, void* ws, size_t ws_bytes,
                               int32_t* status_dev, void* stream);

/* -------------------------------------------------------- row-wise GPTQ
 * The one-sided case B = I of the same solve: with L_B = I every row of W
 * is quantized independently by Algorithm 1 with H = A, i.e. GPTQ ("BaKron:
 * Efficient Quantization with Kronecker-Factored Hessians", Sec. 1: GPTQ's
 * Hessian is X X^T (x) I; Sec. 3.1, Algorithm 1; the GPTQ column of
 * Table 3).  Same arguments, conventions and results as bakron_quantize
 * with LB the identity, without LB; the column terms, column pushes and
 * column chunk products are skipped.  LA: the normalized factor of A (see
 * bakron_factor).  Workspace: bakron_gptq_workspace_size(m, n) bytes.
 */
size_t bakron_gptq_workspace_size(int64_t m, int64_t n);
int bakron_gptq_quantize(const float* W, const float* LA, const float* scales, int bits, int64_t m, int64_t n,
                         int32_t* V, float* Wq, void* ws, size_t ws_bytes, int32_t* status_dev, void* stream);

/* ------------------------------------------------ Hessian factor samples
 * Kronecker factors of a Hessian H = E[a a^T (x) b b^T] from calibration
 * samples ("BaKron: Efficient Quantization with Kronecker-Factored
 * Hessians", Sec. 4.2, App. A.2, App. D):
 *   K-FAC style      A = E[a a^T],          B = E[b b^T];
 *   Shampoo, one power-iteration step from the identity
 *                    A = E[|b|^2 a a^T],    B = E[|a|^2 b b^T];
 *   damping          G + 0.5 mean(diag G) I   (App. D's regularization).
 * Samples are bfloat16 columns, stored feature-major: X is d x N (features
 * x samples), row i at X + i * ldx.  An expectation over several batches of
 * samples is accumulated with beta = 1 and alpha = 1 / (total samples).
 */

/* Workspace bytes of bakron_gram: the samples repacked into 16 KB blocks
 * (128 features x 64 samples, zero-padded), three copies with weights. */
size_t bakron_gram_workspace_size(int64_t d, int64_t N, int weighted);

/* G <- beta G + alpha X diag(w) X^T on the tensor cores (tcgen05; every
 * bf16 product exact; fp32 accumulation over segments of 2048 samples,
 * whose sums are added in fp32, so the rounding error of an entry grows
 * with the segment length and the number of segments, not with N: about
 * 5e-6 relative, Frobenius norm, at 65536 samples).  A packing pass
 * rearranges X into `ws` first; the products then stream 16 KB blocks with
 * bulk copies.
 * X: device, bf16 bit patterns, d x ldx, 16-byte aligned, ldx >= N and a
 *    multiple of 8.
 * w: device, N fp32 per-sample weights, 16-byte aligned, or NULL for ones.
 *    With weights, w_t x_t is split into two bf16 terms (about 2^-17
 *    relative remains) and multiplied in two products.
 * G: device, d x d fp32, written in full (both triangles, symmetric); with
 *    beta != 0 it must be symmetric on entry.  Not aliasing X.
 * ws: device, >= bakron_gram_workspace_size(d, N, w != NULL) bytes, 256-byte
 *    aligned; its contents on entry do not matter.
 * status_dev: device int32, set to 0 or BAKRON_DEV_TIMEOUT.
 * d, N >= 1, d * d < 2^31.  One CTA per 128 x 128 tile of the lower block
 * triangle, enqueued on `stream`.
 */
int bakron_gram(const void* X, int64_t d, int64_t N, int64_t ldx, const float* w, float alpha, float beta, float* G,
                void* ws, size_t ws_bytes, int32_t* status_dev, void* stream);

/* w[t] = |y_t|^2 for the columns of Y (device, bf16, m x ldy, ldy >= N): the
 * weights of one Shampoo step (squares exact, sums in double-float). */
int bakron_sq_norms(const void* Y, int64_t m, int64_t N, int64_t ldy, float* w, void* stream);

/* G <- G + rel * mean(diag G) * I in place (device, d x d fp32; App. D uses
 * rel = 0.5).  One CTA; the trace is summed in double-float. */
int bakron_damp(float* G, int64_t d, float rel, void* stream);

/* ------------------------------------------------- BaKron-antidiagonal
 * Algorithm 3 of "BaKron: Efficient Quantization with Kronecker-Factored
 * Hessians" (Sec. 3.2; the BaKron-antidiag. column of Table 3, equivalent to
 * the iterative YAQA): the anti-diagonals are rounded in order, and after
 * each the errors of the whole anti-diagonal update every later entry,
 *     W~ += L_B Delta L_A^T      (Delta nonzero on one anti-diagonal),
 * m + n - 1 steps and about m^2 n^2 / 4 multiply-adds in all -- the
 * quartic-work baseline BaKron improves on.  Same rounding, arithmetic
 * (double-float) and codes as bakron_quantize (Theorem 3.2), one kernel
 * launch per anti-diagonal on `stream`.  Arguments, results and errors as
 * bakron_quantize; workspace bakron_antidiag_workspace_size(m, n) bytes
 * (8 bytes per weight plus 16 per row).
 */
size_t bakron_antidiag_workspace_size(int64_t m, int64_t n);
int bakron_antidiag_quantize(const float* W, const float* LA, const float* LB, const float* scales, int bits,
                             int64_t m, int64_t n, int32_t* V, float* Wq, void* ws, size_t ws_bytes,
                             int32_t* status_dev, void* stream);

/* -------------------------------------------- alphabets, scales, packing
 * The base quantizer's variants ("BaKron: Efficient Quantization with
 * Kronecker-Factored Hessians", App. D: per-output-feature scales from the
 * row's largest magnitude over the alphabet's reach, optionally shrunk by up
 * to a factor 2 by a mean-squared-error search; Sec. 3.1: integer
 * alphabets).
 */
#define BAKRON_MAX_CODE 32767
#define BAKRON_MAX_SCALE_GRID 256

/* bakron_quantize over an explicit integer alphabet {lo .. hi}:
 *     v_ij = clamp(round_half_even(fp32(W~_ij) / s_i), lo, hi).
 * lo <= 0 <= hi, lo < hi, |lo|, |hi| <= BAKRON_MAX_CODE; the symmetric
 * alphabet {-l .. l} of App. D is lo = -l, hi = l, and bits = b of
 * bakron_quantize is lo = -2^(b-1), hi = 2^(b-1) - 1.  LB may be NULL: then
 * L_B = I and the call is the row-wise GPTQ solve of bakron_gptq_quantize.
 * Every other argument, result and error as in bakron_quantize.
 */
int bakron_quantize_range(const float* W, const float* LA, const float* LB, const float* scales, int lo, int hi,
                          int64_t m, int64_t n, int32_t* V, float* Wq, void* ws, size_t ws_bytes,
                          int32_t* status_dev, void* stream);

/* bakron_quantize_range with one scale per entry (Sec. 3.1: scales "for
 * each row and/or column"):
 *     sigma_ij = fp32(scales[i][j / group] * col_scales[j]),
 *     v_ij = clamp(round_half_even(fp32(W~_ij) / sigma_ij), lo, hi),
 *     Wq_ij = fp32(sigma_ij v_ij).
 * scales: device, m x ceil(n / group) row-major (one scale per run of
 *     `group` consecutive columns of a row), or NULL for ones.
 * group: columns per run; 0 (or >= n) for one scale per row (m scales).
 * col_scales: device, n column scales, or NULL (then sigma_ij is the run's
 *     scale itself, no rounding).
 * All scales > 0 and finite (else BAKRON_DEV_BAD_SCALE in *status_dev).
 * LB may be NULL (L_B = I).  Everything else as bakron_quantize_range.
 */
int bakron_quantize_scaled(const float* W, const float* LA, const float* LB, const float* scales, int64_t group,
                           const float* col_scales, int lo, int hi, int64_t m, int64_t n, int32_t* V, float* Wq,
                           void* ws, size_t ws_bytes, int32_t* status_dev, void* stream);

/* Per-row scales for the alphabet {lo .. hi} (lo < 0 < hi), App. D:
 *     s0_i = fp32(max_j |W_ij| / hi)      (correctly rounded fp32 division),
 *     f_g = fp32(1 - g / (2 (grid - 1))),  g = 0 .. grid-1 (1 down to 1/2),
 *     err_i(s) = sum_j (W_ij - s v_ij)^2,  v_ij = clamp(round_half_even(
 *                fp32(W_ij) / s), lo, hi),
 *     scales[i] = fp32(s0_i f_g) for the g of least err_i, the smallest g
 *                among equal errors.
 * grid = 1: scales[i] = s0_i (no search); 1 <= grid <= BAKRON_MAX_SCALE_GRID.
 * A row without a nonzero entry gets scale 1.  The errors are summed in
 * double-float (each term exact), so two candidates whose errors differ
 * by less than about 1e-12 relative may be ordered either way.
 * group: 0 (or >= n) for one scale per row; else one scale per run of
 *    `group` consecutive columns of each row, each run searched on its own
 *    entries (the last run may be shorter), scales[i][k] row-major,
 *    m x ceil(n / group) -- the layout bakron_quantize_scaled reads.
 * W: device, m x n, finite (a run holding a NaN or infinity gets an
 *    unspecified scale); scales: device, distinct from W.
 * m, n >= 1, m * n < 2^31.  One CTA per run; enqueued on `stream`.
 */
int bakron_row_scales(const float* W, int64_t m, int64_t n, int64_t group, int lo, int hi, int grid, float* scales,
                      void* stream);

/* Packed codes: each code of V (device int32, m x n) as its `bits`-bit two's
 * complement, bits in {2, 4, 8}; code j of row i sits in byte
 * i * ceil(n bits / 8) + floor(j bits / 8) of `out` at bit offset
 * (j bits) mod 8 (little-endian within a byte); each row starts at a byte
 * boundary and a row's unused high bits are zero.  Codes outside
 * {-2^(bits-1) .. 2^(bits-1) - 1} keep only their low `bits` bits.
 * out: device, m * ceil(n bits / 8) bytes.  Enqueued on `stream`.
 */
int bakron_pack_codes(const int32_t* V, int64_t m, int64_t n, int bits, uint8_t* out, void* stream);

/* Diagnostics: bakron_quantize with CUDA events recorded around every
 * kernel launch, for per-kernel timing.  Same arguments and result as
 * bakron_quantize, plus three arrays of BAKRON_KERNEL_CLASSES entries
 * (host memory) receiving, per kernel class, the summed event time in ms,
 * the number of launches and the algorithmic flops (2 per multiply-add of
 * the products L_B E L_A^T the class computes).  Classes: 0 = input
 * check and set-up (including the factors' block exponents), 1 = tile
 * solve (diagonal blocks and the distance-1 neighbours), 2 = mid pushes
 * (single source tiles), 3 = chunk products (batched source tiles, on the
 * tensor cores) -- and 4 = the persistent sweep of
 * bakron_quantize_persistent, which this entry point does not run (always
 * 0 here).  Synchronizes `stream` before it returns; the events add a
 * little time to every launch.
 */
#define BAKRON_KERNEL_CLASSES 5
int bakron_quantize_profile(const float* W, const float* LA, const float* LB, const float* scales, int bits,
                            int64_t m, int64_t n, int32_t* V, float* Wq, void* ws, size_t ws_bytes,
                            int32_t* status_dev, void* stream, double* kernel_ms, int64_t* kernel_launches,
                            double* kernel_flops);

/* Device workspace bytes bakron_quantize_host needs: the device copies of
 * W, LA, LB, scales, V, Wq and the status word, plus
 * bakron_quantize_workspace_size(m, n). */
size_t bakron_quantize_host_workspace_size(int64_t m, int64_t n);

/* Same computation from and to HOST buffers: copies W, LA, LB, scales into
 * `dev_ws`, runs bakron_quantize, copies V and Wq back, and synchronizes
 * `stream` before returning.  scales may be NULL.  *status_host receives
 * the device status word.  dev_ws: device, >= bakron_quantize_host_
 * workspace_size(m, n) bytes, 256-byte aligned.
 */
int bakron_quantize_host(const float* W, const float* LA, const float* LB, const float* scales,
                         int bits, int64_t m, int64_t n, int32_t* V, float* Wq, void* dev_ws,
                         size_t dev_ws_bytes, int32_t* status_host, void* stream);

/* Host-only check of the persistent sweep's task plan for an m x n layer
 * (no GPU involved): every delayed update that the sweep's bands do not
 * apply themselves -- row terms from source tiles at least 3 tiles back,
 * column terms from bands at least 2 bands above ("BaKron", App. B eq. (1):
 * the updates of finished entries are one product L_B E L_A^T restricted
 * to the later ones) -- is carried by exactly one tensor-core task, and no
 * task carries one that the bands apply.  stats (host, 3 entries):
 * [0] number of tasks, [1] the smallest margin in steps, in the ideal
 * schedule, between a task's sources completing and its first target being
 * needed, [2] the number of coverage errors.  Returns BAKRON_OK when there
 * are none, BAKRON_ERR_INVALID_ARG for bad sizes, else 1.
 */
int bakron_sweep_plan_check(int64_t m, int64_t n, int64_t* stats);

/* Host-only check of bakron_quantize's launch schedule for an m x n layer
 * (no GPU involved; the same step numbering, target ranges and chunk
 * candidates as the launches): along every tile column (the column terms
 * L_B[p, i] G[i, q], colpush = 1) and every tile row (the row terms
 * E[p, j] L_A[q, j]) -- together the product L_B E L_A^T restricted to the
 * later entries ("BaKron", App. B eq. (1)) -- each pair of a source tile and
 * a later target tile is carried exactly once, by the target's own solve
 * (adjacent tiles), a mid push or a chunk product; a mid push is complete
 * two steps after its launch, a chunk product `lag` steps after (the solver
 * waits B + 1 = 5 steps; other values test the check); every source is
 * solved before its push is launched and every tile is solved once.
 * colpush = 0 checks the row-wise schedule of bakron_gptq_quantize (L_B = I:
 * no column terms, tile columns as steps).  m, n in 1 .. 2^15.
 * stats (host, 3 entries): [0] pulls and pushes recorded, [1] the smallest
 * number of steps from a chunk product's launch to its first target's solve
 * (-1 without chunk products), [2] errors.  Returns BAKRON_OK when there are
 * none, BAKRON_ERR_INVALID_ARG for bad arguments, else 1.
 */
int bakron_wavefront_plan_check(int64_t m, int64_t n, int colpush, int lag, int64_t* stats);

/* --------------------------------------------------------------- self-test
 * Exercises the device-side timeout path on purpose: one thread waits, with
 * the bounded wait the tensor-core kernels use (about 0.1 s, 2^28 cycles),
 * on an mbarrier that nothing ever arrives on, gives up and sets
 * *status_dev = BAKRON_DEV_TIMEOUT.  Nothing faults or hangs, and the
 * context stays usable.  status_dev: device int32.  Enqueued on `stream`.
 */
int bakron_selftest_wait_timeout(int32_t* status_dev, void* stream);

/* ------------------------------------------------------- no-allocation solve
 * For callers that cannot allocate device memory at all: a plugin inside a
 * host application whose device memory is entirely owned by another
 * allocator, or a latency-critical path that must not call cudaMalloc
 * (which can synchronize the whole device).  The paper has no counterpart;
 * this is an interface convenience.
 *
 * Same computation and arguments as bakron_quantize, without `ws`: the
 * scratch space comes from a fixed array inside the library, of
 * BAKRON_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library holds
 * until the process exits.  The caller still passes (and owns) W, LA, LB,
 * scales, V, Wq and status_dev.  Sizes with
 * bakron_quantize_workspace_size(m, n) > BAKRON_NOALLOC_SCRATCH_BYTES
 * (72 bytes of solver state per weight: up to about 1.16 million weights,
 * e.g. 1024 x 1024) are rejected with
 * BAKRON_ERR_WORKSPACE before anything is enqueued.
 *
 * The first call on a device (and the first call after the device's context
 * was replaced, e.g. by cudaDeviceReset) looks up the array's device address
 * for that device (cudaGetSymbolAddress, with that device current); make
 * that first call before any stream capture.  The call allocates nothing.
 * Every call on a device shares the one array and leaves its contents
 * behind; each call re-initializes what it reads, but calls that overlap on
 * the GPU (other streams, other host threads) race on it: serialize them.
 */
#define BAKRON_NOALLOC_SCRATCH_BYTES ((size_t)80 << 20)
int bakron_quantize_noalloc(const float* W, const float* LA, const float* LB, const float* scales, int bits,
                            int64_t m, int64_t n, int32_t* V, float* Wq, int32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BAKRON_H_ */
