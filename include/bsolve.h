/*
 * bsolve.h -- C ABI of libbsolve.so: batched solution of many independent small dense
 * linear systems A x = b on one GPU (sm_103a).
 *
 * Every entry point solves `batch` independent systems in one asynchronous launch (two
 * when a factor and a solve run apart: a fused call with more than 8 right-hand sides,
 * the row-major reading of the _ex call) on the caller's CUDA stream. All matrix and
 * vector pointers are DEVICE pointers owned by the caller, except those of the
 * *_batched_host calls (host arrays, copied in and out by chunks on two streams); no
 * call allocates memory (the one device scratch, of the _static host call, is placed when
 * the library loads), keeps state for a later call or synchronizes the host. Results are
 * valid once the stream has reached the launch; the per-system `info` array is read back
 * by the caller when it needs it. Calls may run concurrently on different streams and may
 * be captured into CUDA graphs (the _static host call excepted: its entry below says how
 * calls to it may overlap).
 *
 * Batched storage: system s of a batched operand starts at element s * (elements per
 * system); there is no padding between systems. Offsets are 64-bit. (The _ex calls also
 * take the interleaved AoSoA/SoA layouts: bs_options.interleave.)
 *
 * Errors are reported synchronously, before anything is launched:
 *   BS_ERR_INVALID_ARG  null pointer, negative size, a base address not 16-byte aligned,
 *                       or two operands of the call whose byte ranges overlap;
 *   BS_ERR_UNSUPPORTED  a shape, dtype, layout or fill with no kernel instance (there is
 *                       no CPU fallback: the caller chooses another path);
 *   BS_ERR_CUDA         the launch itself failed (bs_last_cuda_error() gives the code).
 * batch == 0 returns BS_OK and launches nothing. Numerical failure of a system (a
 * singular pivot, a minor that is not positive definite) is not an error of the call:
 * it is reported in that system's info entry.
 */
#ifndef BSOLVE_H
#define BSOLVE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BS_API __attribute__((visibility("default")))
#else
#define BS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BS_OK = 0,
  BS_ERR_INVALID_ARG = 1,
  BS_ERR_UNSUPPORTED = 2,
  BS_ERR_CUDA = 3
} bs_status;

typedef enum { BS_FP32 = 0, BS_FP64 = 1 } bs_dtype;

/* Element (r, c) of an n x m operand lives at r*m + c (row-major) or c*n + r
 * (column-major) within its system. */
typedef enum { BS_ROW_MAJOR = 0, BS_COL_MAJOR = 1 } bs_layout;

typedef enum { BS_LOWER = 0, BS_UPPER = 1 } bs_fill;

/*
 * LU factorization with partial pivoting and solve (getrf + getrs), in place.
 *
 * Source: TDLS API, "solver_static.hpp File Reference" (CooperativeLUppSolverStatic),
 * Detailed Description -- right-looking LU with partial pivoting, one system per thread
 * group, rows held in registers, L y = P b folded into the factorization, then U x = y;
 * RUDA docs, "ruSOLVER: small-matrix kernel optimisation" -- lowest-row tie rule,
 * status 0 / first failing pivot, failed outputs zeroed.
 *
 *   A     batch x n x n, in `layout`. On return: L\U of P A in LAPACK format -- row k
 *         holds the unit-lower multipliers of L left of the diagonal and row k of U from
 *         the diagonal on; the diagonal holds the pivots themselves.
 *   B     batch x n x nrhs, same layout as A. On return: X. Systems with info != 0
 *         return X = 0.
 *   ipiv  batch x n int32. ipiv[s*n + k] = 1-based row interchanged with row k at step k
 *         (the LAPACK swap sequence).
 *   info  batch int32. 0 = success; k > 0 = the first step k-1 whose pivot is singular,
 *         i.e. !(|pivot| >= smallest normal number of the dtype) (zero, subnormal or
 *         NaN). The sweep runs to the end with a pivot reciprocal of 1; the factor of
 *         such a system is then unspecified.
 * Pivot choice: the row of largest magnitude in the pivot column, lowest current row
 * on ties. The factorization is of A itself (P A = L U) in both layouts.
 * Supported: dtype FP32/FP64, both layouts, 1 <= n <= 128, 1 <= nrhs <= 65536 (above 8 the
 * call runs as bs_getrf_batched then the solve of bs_getrs_batched, X zeroed where
 * info != 0: the same operations in the same order, so the same bits).
 * stream: a cudaStream_t (0 = the legacy default stream).
 */
BS_API bs_status bs_getrf_getrs_batched(bs_dtype dtype, bs_layout layout, int n, int nrhs,
                                 int64_t batch, void* A, void* B, int32_t* ipiv,
                                 int32_t* info, void* stream);

/*
 * Cholesky factorization and solve (potrf + potrs) of symmetric positive definite
 * systems, in place.
 *
 * Source: cuSolverDx docs, "Cholesky Factorization" (POTRF) -- only the `fill` triangle
 * is read and replaced by the Cholesky factor, the other triangle is untouched; info
 * reports the smallest leading minor that is not positive definite; RUDA docs,
 * "ruSOLVER: small-matrix kernel optimisation" -- failed outputs zeroed.
 *
 *   A     batch x n x n in `layout`; with BS_LOWER only the lower triangle (diagonal
 *         included) is read and replaced by L (A = L L^T), the strict upper triangle is
 *         neither read nor written; with BS_UPPER only the upper triangle is read and
 *         replaced by U (A = U^T U, U = L^T: the same operations on mirrored entries),
 *         the strict lower triangle is neither read nor written.
 *   B     batch x n x nrhs, same layout as A. On return: X (zero where info != 0).
 *   info  batch int32. 0 = success; k > 0 = the leading minor of order k is not positive
 *         definite (the k-th diagonal of the factorization is not > 0, NaN included).
 *         The factor from column k-1 on is then unspecified.
 * Supported: dtype FP32/FP64, both layouts, fill BS_LOWER or BS_UPPER, 1 <= n <= 256,
 * 1 <= nrhs <= 65536 (above 8 right-hand sides, and for every n > 128:
 * bs_potrf_batched then the solve of bs_potrs_batched, X zeroed where info != 0). For
 * 128 < n <= 256 the factor runs on a cluster of four CTAs per system, the 32 x 32 tiles
 * of the triangle spread over their shared memory and read across the cluster
 * (cuSolverDx docs, "Cholesky Factorization": the cluster tiling beyond one CTA); the
 * results are the same operations in the same order as for any other n.
 */
BS_API bs_status bs_potrf_potrs_batched(bs_dtype dtype, bs_layout layout, bs_fill fill, int n,
                                 int nrhs, int64_t batch, void* A, void* B, int32_t* info,
                                 void* stream);

/*
 * Block-tridiagonal symmetric positive definite solve by the block-Cholesky
 * (block-Thomas) sweep (bdsv = bdsv_factor + bdsv_solve), in place.
 *
 * Source: GLASS API reference, "Block-tridiagonal Ops", sections "Block-tridiagonal
 * matrix-vector product" (strip and padded-vector layouts) and "Direct solve
 * (glass::bdsv)" (the factorization and the two sweeps).
 *
 *   strips    batch x num_block_rows x block_size x (3*block_size): block-row br of a
 *             system is a row-major strip [L | D | R]; entry (y, x) of slot s (LEFT 0,
 *             MAIN 1, RIGHT 2) at strip[y*3*bs + s*bs + x]. D is read through its lower
 *             triangle, L_br for br >= 1; L_0 and every RIGHT slot are never read.
 *             On return: MAIN <- F_k lower triangle (its strict upper triangle keeps D_k),
 *             LEFT <- E_k for k >= 1; RIGHT slots untouched.
 *             F_0 = chol(D_0); E_k = L_k F_{k-1}^{-T}; F_k = chol(D_k - E_k E_k^T).
 *   x_padded  batch x (num_block_rows + 2)*block_size: block-row br at (br+1)*block_size.
 *             On entry the interior holds b, on return x; the two pad blocks are neither
 *             read nor written.
 *   info      batch int32. 0 = success; k > 0 = global index br*bs + j + 1 of the first
 *             diagonal of the sweep that is not > 0 (the dense Cholesky factor of the
 *             assembled matrix fails at the same minor). x is then zero and the strips
 *             from that knot on are unspecified.
 * Supported: dtype FP32/FP64, 1 <= block_size <= 8, num_block_rows >= 1.
 */
BS_API bs_status bs_bdsv_batched(bs_dtype dtype, int num_block_rows, int block_size, int64_t batch,
                          void* strips, void* x_padded, int32_t* info, void* stream);

/*
 * Contract variants of the two fused dense calls.
 *
 * Source: TDLS API, "solver_static.hpp File Reference", Detailed Description
 * (Config.relative_pivot_threshold: 1 keeps the choice of MAGMA and LAPACK, a smaller value
 * keeps the row in place more often); RUDA docs, "ruSOLVER: small-matrix kernel
 * optimisation" (unchanged numerical and failure contract: status codes and failed
 * outputs).
 *
 *   pivot_threshold  tau in (0, 1] (LU only). At step k, with m the magnitude partial
 *                    pivoting finds, the row in place stays the pivot when
 *                    |a_kk| >= tau * m (the product rounded in the dtype); otherwise the
 *                    first maximum is taken. 1 = partial pivoting. Every multiplier then
 *                    obeys |l_ik| <= 1/tau.
 *   status_contract  BS_CONTRACT_DEFAULT: as the plain calls. BS_CONTRACT_RUDA: info is
 *                    0 success, k > 0 the first failing pivot or minor, -1 a non-finite
 *                    entry in A or B, -2 (Cholesky) A not exactly symmetric (the whole
 *                    matrix is read), -3 a non-finite entry of the factor or X after a
 *                    sweep without a failing pivot; a failed system (info != 0) returns
 *                    its factor (Cholesky: the fill triangle) and X as zeros and, for LU,
 *                    every ipiv entry as -1.
 *   transposed_factor  0 or 1 (LU only; TDLS API, "solver_static.hpp File Reference", the
 *                    row-major layout: the solver factors S, the stored array read
 *                    column-major). 1 with BS_ROW_MAJOR factors S = A^T in place,
 *                    P A^T = L U (ipiv: LAPACK's 1-based swap sequence of that factor,
 *                    i.e. interchanges of columns of A), and solves the mirror
 *                    U^T z = b, L^T w = z, x = P^T w; X is zeros where info != 0. A then
 *                    holds the factor of A^T in the column-major reading. With
 *                    BS_COL_MAJOR, S = A and the call is the plain one. Runs as a factor
 *                    launch and a solve launch, for 1 <= n <= 128, 1 <= nrhs <= 65536;
 *                    with BS_CONTRACT_RUDA it is BS_ERR_UNSUPPORTED (the contract zeroes
 *                    a failed system inside the one fused kernel).
 *   interleave       the batched layout (TDLS API, "solver_static.hpp File Reference":
 *                    element e of a system at base[e * stride]). 0 or 1: AoS, system s
 *                    at s * size (the plain layout). W > 1: AoSoA, the systems in blocks
 *                    of W, element e of system s (e its offset in the system's own storage
 *                    order, size = n*n for A, n*nrhs for B, n for ipiv) at
 *                    (s / W) * W * size + e * W + s % W; W >= batch is SoA. A, B and
 *                    ipiv then hold ceil(batch / W) * W systems each (the slots of the last
 *                    block past the batch are neither read nor written); info keeps one
 *                    entry per system. Cholesky: n <= 128. nrhs <= 8, except with
 *                    transposed_factor (the solve there is a launch of its own, taking 8
 *                    columns at a time: nrhs <= 65536). It combines with the threshold, the
 *                    RUDA contract (one system per CTA), transposed_factor and scaling;
 *                    negative: BS_ERR_INVALID_ARG.
 *   scaling          0 or 1 (LU only; RUDA docs, unchanged numerical contract: the LU keeps
 *                    the scaling by the whole matrix's largest magnitude and restores U's
 *                    scale at the end). 1: with m = max |a_ij| finite and positive, A is
 *                    divided by m before the sweep (each entry rounded once), U (diagonal
 *                    included) is multiplied by m after it, and the back substitution uses
 *                    the restored U (reciprocals of its diagonal recomputed; 1 for one below
 *                    the smallest normal number); a non-finite entry or a zero matrix leaves
 *                    the system unscaled; info reports the scaled sweep's pivots. One
 *                    system per CTA; combines with the threshold, the RUDA contract,
 *                    interleaving and transposed_factor (there S, the stored array read
 *                    column-major, is what is scaled).
 * opts == NULL or default options run the plain call. Thresholds and the RUDA contract
 * run one system per CTA for every n (1 <= n <= 128, 1 <= nrhs <= 8); results equal the
 * CPU oracle's bit for bit. A threshold outside (0, 1], an unknown contract or a
 * transposed_factor other than 0 or 1 is BS_ERR_INVALID_ARG.
 */
typedef enum { BS_CONTRACT_DEFAULT = 0, BS_CONTRACT_RUDA = 1 } bs_contract;

typedef struct {
  double pivot_threshold; /* in (0, 1]; 1 = partial pivoting */
  int status_contract;    /* a bs_contract */
  int transposed_factor;  /* 1: TDLS's row-major reading (factor of A^T, mirror solve) */
  int64_t interleave;     /* batched layout: 0/1 AoS, W > 1 AoSoA blocks of W (SoA: >= batch) */
  int scaling;            /* 1: RUDA's max-abs scaling with U's scale restored (LU) */
} bs_options;

BS_API bs_status bs_getrf_getrs_batched_ex(bs_dtype dtype, bs_layout layout, int n, int nrhs,
                                           int64_t batch, void* A, void* B, int32_t* ipiv,
                                           int32_t* info, const bs_options* opts, void* stream);
BS_API bs_status bs_potrf_potrs_batched_ex(bs_dtype dtype, bs_layout layout, bs_fill fill, int n,
                                           int nrhs, int64_t batch, void* A, void* B,
                                           int32_t* info, const bs_options* opts, void* stream);

/*
 * Factor once, solve per right-hand side: the two halves of the fused calls above.
 *
 * Source: GLASS API reference, "Block-tridiagonal Ops", "Direct solve (glass::bdsv)"
 * (bdsv_factor, bdsv_solve: "reusable: factor once, call this per right-hand side");
 * TDLS API, "solver_static.hpp File Reference", Detailed Description (the substitution as
 * a step of its own after the factorization).
 *
 * The factor calls leave A (or the strips), ipiv and info exactly as the fused call does;
 * the solve calls, given that factor, leave exactly the fused call's X wherever info == 0
 * (same operations in the same order). The solve calls take no info: with a factor whose
 * info != 0 their X is unspecified (the fused calls return zeros there).
 *
 * bs_getrf_batched:  A (batch x n x n, `layout`) <- L\U, ipiv, info as bs_getrf_getrs_batched.
 * bs_getrs_batched:  LU, ipiv from bs_getrf_batched (read only; an ipiv entry outside 1..n
 *                    swaps nothing); B (batch x n x nrhs, same layout) <- X. B must not
 *                    overlap LU or ipiv.
 * bs_potrf_batched:  A <- L or U in the `fill` triangle (the other triangle neither read
 *                    nor written), info as bs_potrf_potrs_batched.
 * bs_potrs_batched:  the factor from bs_potrf_batched with the same fill (read only, its
 *                    triangle only); B <- X.
 * bs_bdsv_factor_batched: strips <- F_k (MAIN, lower), E_k (LEFT); info as bs_bdsv_batched.
 * bs_bdsv_solve_batched:  strips from bs_bdsv_factor_batched (read only); interior of
 *                    x_padded: b on entry, x on return (pads neither read nor written).
 * Supported: as the fused calls (getrf: 1 <= n <= 128; potrf: 1 <= n <= 256; getrs:
 * 1 <= n <= 128, potrs: 1 <= n <= 256, 1 <= nrhs <= 65536, taken 8 columns at a time;
 * bdsv: 1 <= block_size <= 8), FP32/FP64, both layouts, both fills.
 */
BS_API bs_status bs_getrf_batched(bs_dtype dtype, bs_layout layout, int n, int64_t batch, void* A,
                                  int32_t* ipiv, int32_t* info, void* stream);
BS_API bs_status bs_getrs_batched(bs_dtype dtype, bs_layout layout, int n, int nrhs, int64_t batch,
                                  const void* LU, const int32_t* ipiv, void* B, void* stream);
BS_API bs_status bs_potrf_batched(bs_dtype dtype, bs_layout layout, bs_fill fill, int n,
                                  int64_t batch, void* A, int32_t* info, void* stream);
BS_API bs_status bs_potrs_batched(bs_dtype dtype, bs_layout layout, bs_fill fill, int n, int nrhs,
                                  int64_t batch, const void* L, void* B, void* stream);
BS_API bs_status bs_bdsv_factor_batched(bs_dtype dtype, int num_block_rows, int block_size,
                                        int64_t batch, void* strips, int32_t* info, void* stream);
BS_API bs_status bs_bdsv_solve_batched(bs_dtype dtype, int num_block_rows, int block_size,
                                       int64_t batch, const void* strips, void* x_padded,
                                       void* stream);

/*
 * The split calls with options: the factor and the solve of the LU and Cholesky paths on
 * the interleaved batched layouts and, for LU, under TDLS's row-major reading and a pivot
 * threshold.
 *
 * Source: TDLS API, "solver_static.hpp File Reference" (the interleaved batched layouts;
 * the row-major reading; the substitution as a step of its own); RUDA docs (the pivot
 * threshold).
 *
 * Arguments as the split calls above, plus opts (NULL: the plain call), read as the fused
 * _ex calls read them:
 *   interleave         every batched operand (A, B, ipiv) in the layout of that name;
 *                      held ceil(batch / W) * W systems each; info one entry per system.
 *   transposed_factor  1 with BS_ROW_MAJOR: bs_getrf_batched_ex factors S (the array read
 *                      column-major), bs_getrs_batched_ex runs the mirror solve with that
 *                      factor. With BS_COL_MAJOR it changes nothing. Cholesky:
 *                      BS_ERR_UNSUPPORTED.
 *   pivot_threshold    bs_getrf_batched_ex: the threshold rule of the fused call. The solve
 *                      and the Cholesky calls accept any valid value and ignore it.
 *   status_contract    BS_CONTRACT_RUDA: BS_ERR_UNSUPPORTED (a fused-call contract).
 *   scaling            1: BS_ERR_UNSUPPORTED (a fused-call option: the solve uses the
 *                      restored U with recomputed reciprocals).
 * Results: the factor calls leave info, ipiv and, on every system with info == 0, A
 * exactly as the fused _ex call with the same options (a Cholesky system that failed may
 * hold other partial values: interleaved factors of n <= 32 run on another kernel than
 * the fused call's); the solve calls, given that factor, leave the fused call's X wherever
 * info == 0 (with a failed factor X is unspecified). Interleaved or threshold factors run
 * one system per CTA; interleaved or mirror solves one system per warp in shared memory.
 * Supported: LU 1 <= n <= 128; Cholesky 1 <= n <= 256 on the plain layout, n <= 128
 * interleaved; 1 <= nrhs <= 65536.
 */
BS_API bs_status bs_getrf_batched_ex(bs_dtype dtype, bs_layout layout, int n, int64_t batch,
                                     void* A, int32_t* ipiv, int32_t* info,
                                     const bs_options* opts, void* stream);
BS_API bs_status bs_getrs_batched_ex(bs_dtype dtype, bs_layout layout, int n, int nrhs,
                                     int64_t batch, const void* LU, const int32_t* ipiv, void* B,
                                     const bs_options* opts, void* stream);
BS_API bs_status bs_potrf_batched_ex(bs_dtype dtype, bs_layout layout, bs_fill fill, int n,
                                     int64_t batch, void* A, int32_t* info,
                                     const bs_options* opts, void* stream);
BS_API bs_status bs_potrs_batched_ex(bs_dtype dtype, bs_layout layout, bs_fill fill, int n,
                                     int nrhs, int64_t batch, const void* L, void* B,
                                     const bs_options* opts, void* stream);

/*
 * Block-tridiagonal matrix-vector product y = A x (glass::bdmv).
 *
 * Source: GLASS API reference, "Block-tridiagonal Ops", section "Block-tridiagonal
 * matrix-vector product (glass::bdmv)" -- strips [L | D | R], padded vectors, block-row br
 * reads the window x_padded[br*bs, br*bs + 3*bs) and writes y_padded[(br+1)*bs + row].
 *
 *   strips    as bs_bdsv_batched, read only; all three blocks are read as stored (the
 *             caller keeps the pad blocks of x_padded zero, so that L_0 and R_{nbr-1}
 *             multiply zeros).
 *   x_padded  batch x (num_block_rows + 2)*block_size, read only.
 *   y_padded  same shape; the interior receives A x, the two pad blocks are not written.
 *             Must not overlap strips or x_padded (BS_ERR_INVALID_ARG when it does).
 * Each entry is one dot product over its strip row in increasing column order, one fused
 * multiply-add per term, from zero (the pages fix no order; the result does not depend on
 * the launch configuration).
 * Supported: dtype FP32/FP64, 1 <= block_size <= 8, num_block_rows >= 1.
 */
BS_API bs_status bs_bdmv_batched(bs_dtype dtype, int num_block_rows, int block_size, int64_t batch,
                                 const void* strips, const void* x_padded, void* y_padded,
                                 void* stream);

/*
 * The second form of the same page's matvec: one pass that stores the product into two
 * padded outputs (the page's use: z = p = A r at the start of a conjugate-gradient
 * solve). Arguments as bs_bdmv_batched, plus
 *   y2_padded  a second output of y_padded's shape receiving the same values (the pad
 *              blocks not written); must not be null (when batch > 0) and must overlap
 *              none of strips, x_padded and y_padded (BS_ERR_INVALID_ARG).
 * Both outputs hold exactly the values bs_bdmv_batched writes.
 */
BS_API bs_status bs_bdmv2_batched(bs_dtype dtype, int num_block_rows, int block_size,
                                  int64_t batch, const void* strips, const void* x_padded,
                                  void* y_padded, void* y2_padded, void* stream);

/* Human-readable name of a status code (a static string). */
BS_API const char* bs_status_string(bs_status status);

/*
 * Host-resident batches: the fused calls on arrays in host memory, copied in and out by
 * the library in chunks that overlap the copies with the solves.
 *
 * Source: the fused calls above (same operands, layouts, results and status contract);
 * RUDA docs, "ruSOLVER: small-matrix kernel optimisation" (a user call validates on the
 * host before anything is submitted; an empty batch submits nothing).
 *
 *   A, B, ipiv, info, strips, x_padded  HOST arrays in the layouts of the fused calls,
 *             read and overwritten in place with the results. Page-locked (pinned) memory
 *             is what lets the copies run asynchronously and overlap; pageable memory
 *             works but the copies then serialise.
 *   work      DEVICE workspace of at least bs_*_host_workspace(...) bytes, 256-byte
 *             aligned, owned by the caller (the library allocates nothing). Two slots of
 *             one chunk of every operand.
 *   chunk     systems per chunk (>= 1); chunk c runs its host-to-device copies, its solve
 *             and its device-to-host copies on stream (c % 2 ? stream1 : stream0), in
 *             workspace slot c % 2, so the two streams alternate and overlap (stream1 may
 *             equal stream0: correct, no overlap).
 * The call enqueues and returns: the results are in the host arrays once both streams
 * have completed (e.g. cudaStreamSynchronize on each); the host arrays and the workspace
 * must stay valid until then. Errors: the fused calls' (shape, dtype, null pointers),
 * plus BS_ERR_INVALID_ARG for chunk < 1 or a workspace too small or misaligned. A CUDA
 * error of a copy returns BS_ERR_CUDA; chunks already enqueued then complete or fail on
 * their own. The *_host_workspace queries return 0 for invalid sizes.
 */
BS_API size_t bs_getrf_getrs_host_workspace(bs_dtype dtype, int n, int nrhs, int64_t chunk);
BS_API bs_status bs_getrf_getrs_batched_host(bs_dtype dtype, bs_layout layout, int n, int nrhs,
                                             int64_t batch, void* A, void* B, int32_t* ipiv,
                                             int32_t* info, void* work, size_t work_bytes,
                                             int64_t chunk, void* stream0, void* stream1);
/*
 * bs_getrf_getrs_batched_host without a workspace argument, for callers that cannot
 * allocate device memory themselves (code that must not call cudaMalloc, e.g. because it
 * runs under an allocator or a memory budget that it does not control). The paper has no
 * counterpart: the pages solve device-resident batches only.
 *
 * The library's own static device scratch (64 MiB, placed by the driver when the library
 * loads; the call allocates nothing) holds the two chunk slots at fixed offsets, 0 and
 * 32 MiB, and the chunk is the requested one halved until one slot fits 32 MiB
 * (BS_ERR_UNSUPPORTED if a single system does not fit). The first call on a device looks
 * up the scratch's device address on that device (cudaGetSymbolAddress) and keeps it;
 * make that first call before any stream capture on that device.
 *
 * One scratch serves the whole process and keeps the last call's contents (every byte a
 * call reads there it has copied in first). Calls queued one after another on the same
 * two streams, passed in the same order, are kept apart by stream order whatever their
 * shapes; any other pair of calls whose work overlaps on the GPU (other streams, the two
 * streams swapped, several host threads) races on the scratch and corrupts results:
 * synchronize between them. Otherwise as bs_getrf_getrs_batched_host.
 */
BS_API bs_status bs_getrf_getrs_batched_host_static(bs_dtype dtype, bs_layout layout, int n,
                                                    int nrhs, int64_t batch, void* A, void* B,
                                                    int32_t* ipiv, int32_t* info, int64_t chunk,
                                                    void* stream0, void* stream1);
BS_API size_t bs_potrf_potrs_host_workspace(bs_dtype dtype, int n, int nrhs, int64_t chunk);
BS_API bs_status bs_potrf_potrs_batched_host(bs_dtype dtype, bs_layout layout, bs_fill fill,
                                             int n, int nrhs, int64_t batch, void* A, void* B,
                                             int32_t* info, void* work, size_t work_bytes,
                                             int64_t chunk, void* stream0, void* stream1);
BS_API size_t bs_bdsv_host_workspace(bs_dtype dtype, int num_block_rows, int block_size,
                                     int64_t chunk);
BS_API bs_status bs_bdsv_batched_host(bs_dtype dtype, int num_block_rows, int block_size,
                                      int64_t batch, void* strips, void* x_padded,
                                      int32_t* info, void* work, size_t work_bytes,
                                      int64_t chunk, void* stream0, void* stream1);

/* The CUDA error code of the last BS_ERR_CUDA returned on this host thread (0 if none). */
BS_API int bs_last_cuda_error(void);

/* 1 if the call with these arguments has a kernel instance, else 0 (no launch). */
BS_API int bs_getrf_getrs_supported(bs_dtype dtype, bs_layout layout, int n, int nrhs);
BS_API int bs_potrf_potrs_supported(bs_dtype dtype, bs_layout layout, bs_fill fill, int n,
                                     int nrhs);
BS_API int bs_bdsv_supported(bs_dtype dtype, int num_block_rows, int block_size);

/* Library ABI version (major*10000 + minor*100 + patch). */
BS_API int bs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSOLVE_H */
