// Host-side launchers of the CUDA kernels (internal to libbsolve.so).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace bsolve {

// LU + solve, rows in registers, 1 <= n <= 32, 0 <= nrhs <= 8 (0: factor only). The
// LU and Cholesky launchers below take nrhs = 0 the same way.
template <typename T>
cudaError_t launch_lu_reg(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                          int32_t* ipiv, int32_t* info, cudaStream_t stream);
// The same on the interleaved batched layout (element e of system s at
// (s / ilv) * ilv * size + e * ilv + s % ilv for A, B and ipiv), 1 <= nrhs <= 8.
template <typename T>
cudaError_t launch_lu_reg_il(int layout, int n, int nrhs, int64_t batch, int64_t ilv, T* A, T* B,
                             int32_t* ipiv, int32_t* info, cudaStream_t stream);

// LU + solve, one block of four warps per system in shared memory, 1 <= n <= 128, 0 <= nrhs <= 8.
template <typename T>
cudaError_t launch_lu_smem(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                           int32_t* ipiv, int32_t* info, cudaStream_t stream);

// The same with the options of the _ex calls: TDLS threshold tau in (0, 1], RUDA status
// contract (ruda != 0); any 1 <= n <= 128.
// LU + solve for FP32, 8 < n <= 16, nrhs <= 8 (0: factor only), two rows per lane and
// four systems per warp; ilv: the element stride of an interleaved batched layout (1: plain).
cudaError_t launch_lu_rows2(int layout, int n, int nrhs, int64_t batch, float* A, float* B,
                            int32_t* ipiv, int32_t* info, cudaStream_t stream, int64_t ilv = 1);

template <typename T>
cudaError_t launch_lu_smem_ex(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                              int32_t* ipiv, int32_t* info, double tau, int ruda,
                              cudaStream_t stream, int64_t ilv = 1, int scale = 0);

// Solve with a stored factor: getrs (L\U and the 1-based swap sequence of getrf) and
// potrs (Cholesky factor), 1 <= n <= 128.
// Any nrhs >= 1 (a register tier's worth at a time). zinfo (may be null): X = 0 where
// zinfo[s] != 0.
// ilv: the element stride of an interleaved batched layout (1: the plain layout; > 1:
// n <= 128, one warp per system).
template <typename T>
cudaError_t launch_getrs(int layout, int n, int nrhs, int64_t batch, const T* LU,
                         const int32_t* ipiv, T* B, const int32_t* zinfo, cudaStream_t stream,
                         int64_t ilv = 1);
template <typename T>
cudaError_t launch_potrs(int layout, int n, int nrhs, int64_t batch, const T* L, T* B,
                         const int32_t* zinfo, cudaStream_t stream, int64_t ilv = 1);
// potrs for FP64, 1 <= n <= 32, nrhs == 1: one system per lane, the factor streamed by
// columns through shared memory (layout bit 0: the factor's storage order).
cudaError_t launch_potrs_lane(int layout, int n, int nrhs, int64_t batch, const double* L,
                              double* B, const int32_t* zinfo, cudaStream_t stream);

// The mirror solve of the row-major reading (U^T z = b, L^T w = z, x = P^T w) with the LU
// factor of S, the stored array read column-major; layout packs S's order (bit 0) and B's.
template <typename T>
cudaError_t launch_getrs_mirror(int layout, int n, int nrhs, int64_t batch, const T* S,
                                const int32_t* ipiv, T* B, const int32_t* zinfo,
                                cudaStream_t stream, int64_t ilv = 1);

// The Cholesky launchers (chol_smem, chol_sys, potrs) take a packed storage-order code:
// bit 0 for A (or the factor), bit 1 for B; upper fill is passed as the lower fill of A in
// the other order.
// Lower Cholesky + solve, one warp per system in shared memory, 1 <= n <= 128.
template <typename T>
cudaError_t launch_chol_smem(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                             int32_t* info, cudaStream_t stream);

// The same under the RUDA status contract (ruda != 0): -1 non-finite input, -2 input
// not symmetric (the whole matrix is read), -3 non-finite result; failures zeroed.
template <typename T>
cudaError_t launch_chol_smem_ex(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                                int32_t* info, int ruda, cudaStream_t stream, int64_t ilv = 1);

// Lower Cholesky factor (potrf) for 128 < n <= 256 on a cluster of four CTAs, the tiles
// of one system spread over their shared memory; layout bit 0: A's storage order.
template <typename T>
cudaError_t launch_chol_cluster(int layout, int n, int64_t batch, T* A, int32_t* info,
                                cudaStream_t stream);
// potrs for 128 < n <= 256, any nrhs >= 1: one CTA per system (packed storage-order code).
template <typename T>
cudaError_t launch_potrs_big(int layout, int n, int nrhs, int64_t batch, const T* L, T* B,
                             const int32_t* zinfo, cudaStream_t stream);

// Lower Cholesky + solve, sixteen systems per block in lockstep, 1 <= n <= 32.
template <typename T>
cudaError_t launch_chol_sys(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                            int32_t* info, cudaStream_t stream, int64_t ilv = 1);

// Block-tridiagonal block-Cholesky sweep, one thread per system, 1 <= bs <= 8.
template <typename T>
cudaError_t launch_bdsv(int nbr, int bs, int64_t batch, T* strips, T* xpad, int32_t* info,
                        cudaStream_t stream);

// The factor sweep alone, and the substitutions alone on factored strips.
template <typename T>
cudaError_t launch_bdsv_factor(int nbr, int bs, int64_t batch, T* strips, int32_t* info,
                               cudaStream_t stream);
template <typename T>
cudaError_t launch_bdsv_solve(int nbr, int bs, int64_t batch, const T* strips, T* xpad,
                              cudaStream_t stream);

// Block-tridiagonal matrix-vector product on padded vectors, 1 <= bs <= 8; ypad2, when
// not null, receives the same product too.
template <typename T>
cudaError_t launch_bdmv(int nbr, int bs, int64_t batch, const T* strips, const T* xpad, T* ypad,
                        T* ypad2, cudaStream_t stream);

// Shared memory one system needs in the shared-memory kernels.
size_t lu_cta_bytes(int n, int nrhs, int elem_size);
size_t chol_smem_bytes(int n, int nrhs, int elem_size);
size_t chol_sys_bytes(int n, int nrhs, int elem_size);

}  // namespace bsolve
