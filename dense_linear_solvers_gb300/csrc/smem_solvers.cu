// LU with partial pivoting and lower Cholesky, one warp per system, with the system
// resident in shared memory (n <= 64).
//
// The system is held as one n x P row-major tile M = [A | B] (P = n + nrhs rounded up to
// an odd number of elements, so that walking down a column touches distinct banks).
// Every step of the right-looking factorization spreads its trailing update over the
// 32 lanes element by element (a column-major walk of the trailing block), so that the
// warp's instructions stay busy however small the trailing block gets; this matters on
// a part whose FP64 pipe charges a whole warp instruction whatever its active lanes.
//
// LU: physical row interchanges in LAPACK order (TDLS API, "solver_static.hpp File
// Reference", Detailed Description: physical interchanges choose the same pivots and run
// the same operations as the logical ones), pivot search with integer magnitude keys
// and the lowest-row tie rule, L y = P b folded into the factorization, then U x = y.
// Cholesky: right-looking lower factorization (cuSolverDx docs, "Cholesky
// Factorization": only the lower triangle is read and written), the forward solve
// folded in, then L^T x = y.
// The arithmetic is the CPU oracle's, operation by operation.
#include "common.cuh"
#include "kernels.h"

namespace bsolve {
namespace {

__host__ __device__ inline int odd_pitch(int w) { return w | 1; }

template <typename T>
__device__ __forceinline__ void load_system(const T* __restrict__ A, const T* __restrict__ B,
                                            T* M, int n, int nrhs, int P, int layout,
                                            bool lower_only, int lane) {
  if (layout == kRowMajor) {
    for (int i = 0; i < n; ++i) {
      const int jend = lower_only ? i + 1 : n;
      for (int j = lane; j < jend; j += 32) M[i * P + j] = A[i * n + j];
    }
    for (int e = lane; e < n * nrhs; e += 32) {
      const int i = e / nrhs, c = e - i * nrhs;
      M[i * P + n + c] = B[e];
    }
  } else {
    for (int j = 0; j < n; ++j)
      for (int i = (lower_only ? j : 0) + lane; i < n; i += 32) M[i * P + j] = A[j * n + i];
    for (int c = 0; c < nrhs; ++c)
      for (int i = lane; i < n; i += 32) M[i * P + n + c] = B[c * n + i];
  }
}

template <typename T>
__device__ __forceinline__ void store_system(T* __restrict__ A, T* __restrict__ B, const T* M,
                                             int n, int nrhs, int P, int layout,
                                             bool lower_only, bool zero_x, int lane) {
  if (layout == kRowMajor) {
    for (int i = 0; i < n; ++i) {
      const int jend = lower_only ? i + 1 : n;
      for (int j = lane; j < jend; j += 32) A[i * n + j] = M[i * P + j];
    }
    for (int e = lane; e < n * nrhs; e += 32) {
      const int i = e / nrhs, c = e - i * nrhs;
      B[e] = zero_x ? T(0) : M[i * P + n + c];
    }
  } else {
    for (int j = 0; j < n; ++j)
      for (int i = (lower_only ? j : 0) + lane; i < n; i += 32) A[j * n + i] = M[i * P + j];
    for (int c = 0; c < nrhs; ++c)
      for (int i = lane; i < n; i += 32) B[c * n + i] = zero_x ? T(0) : M[i * P + n + c];
  }
}

template <typename T>
__global__ void __launch_bounds__(32)
lu_smem_kernel(int n, int nrhs, int layout, int64_t batch, T* __restrict__ A,
               T* __restrict__ B, int32_t* __restrict__ ipiv, int32_t* __restrict__ info) {
  using Key = typename Traits<T>::Key;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x;
  const int64_t s = blockIdx.x;
  if (s >= batch) return;
  const int P = odd_pitch(n + nrhs);
  T* M = reinterpret_cast<T*>(smem_raw);
  T* rcp = M + n * P;
  int* piv = reinterpret_cast<int*>(rcp + n);

  A += s * n * n;
  B += s * n * nrhs;
  load_system<T>(A, B, M, n, nrhs, P, layout, false, lane);
  __syncwarp();

  int inf = 0;
  for (int k = 0; k < n; ++k) {
    // pivot search over rows k..n-1 of column k; a lane keeps its first maximum
    Key best = 0;
    int bi = 0x7FFFFFFF;
    for (int i = k + lane; i < n; i += 32) {
      const Key key = pivot_key<T>(M[i * P + k], i == k);
      if (key > best) {
        best = key;
        bi = i;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const Key ob = shfl_xor_key(best, off, 32);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
      }
    }
    const int p = bi;
    const bool ok = pivot_ok<T>(best);
    if (!ok && inf == 0) inf = k + 1;
    if (lane == 0) piv[k] = p + 1;
    if (p != k) {
      for (int j = lane; j < n + nrhs; j += 32) {
        const T t = M[k * P + j];
        M[k * P + j] = M[p * P + j];
        M[p * P + j] = t;
      }
    }
    __syncwarp();
    const T r = ok ? T(1) / M[k * P + k] : T(1);
    if (lane == 0) rcp[k] = r;
    for (int i = k + 1 + lane; i < n; i += 32) M[i * P + k] = M[i * P + k] * r;
    __syncwarp();
    // rank-1 update of rows k+1..n-1, columns k+1..n+nrhs-1, walked column by column
    const int m = n - k - 1;
    const int w = n + nrhs - k - 1;
    if (m > 0) {
      const int total = m * w;
      const int dq = 32 / m, dr = 32 - dq * m;
      int ii = lane % m, jj = lane / m;
      for (int e = lane; e < total; e += 32) {
        const int i = k + 1 + ii, j = k + 1 + jj;
        M[i * P + j] = fma_rn<T>(-M[i * P + k], M[k * P + j], M[i * P + j]);
        ii += dr;
        jj += dq;
        if (ii >= m) {
          ii -= m;
          ++jj;
        }
      }
    }
    __syncwarp();
  }
  // U x = y
  for (int i = n - 1; i >= 0; --i) {
    const T r = rcp[i];
    for (int c = lane; c < nrhs; c += 32) M[i * P + n + c] = M[i * P + n + c] * r;
    __syncwarp();
    const int total = i * nrhs;
    for (int e = lane; e < total; e += 32) {
      const int c = e / i, i2 = e - c * i;
      M[i2 * P + n + c] = fma_rn<T>(-M[i2 * P + i], M[i * P + n + c], M[i2 * P + n + c]);
    }
    __syncwarp();
  }
  store_system<T>(A, B, M, n, nrhs, P, layout, false, inf != 0, lane);
  for (int k = lane; k < n; k += 32) ipiv[s * n + k] = piv[k];
  if (lane == 0) info[s] = inf;
}

template <typename T>
__global__ void __launch_bounds__(32)
chol_smem_kernel(int n, int nrhs, int layout, int64_t batch, T* __restrict__ A,
                 T* __restrict__ B, int32_t* __restrict__ info) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x;
  const int64_t s = blockIdx.x;
  if (s >= batch) return;
  const int P = odd_pitch(n + nrhs);
  T* M = reinterpret_cast<T*>(smem_raw);
  T* rcp = M + n * P;

  A += s * n * n;
  B += s * n * nrhs;
  load_system<T>(A, B, M, n, nrhs, P, layout, true, lane);
  __syncwarp();

  int inf = 0;
  for (int k = 0; k < n; ++k) {
    const T d = M[k * P + k];
    if (!(d > T(0))) {
      inf = k + 1;
      break;
    }
    const T l = sqrt(d);
    const T r = T(1) / l;
    __syncwarp();
    if (lane == 0) {
      M[k * P + k] = l;
      rcp[k] = r;
    }
    for (int i = k + 1 + lane; i < n; i += 32) M[i * P + k] = M[i * P + k] * r;
    for (int c = lane; c < nrhs; c += 32) M[k * P + n + c] = M[k * P + n + c] * r;
    __syncwarp();
    // lower trailing triangle, walked column by column: column j holds rows j..n-1
    {
      int j = k + 1, i = k + 1 + lane;
      while (j < n && i >= n) {
        i -= n;
        ++j;
        i += j;
      }
      while (j < n) {
        M[i * P + j] = fma_rn<T>(-M[i * P + k], M[j * P + k], M[i * P + j]);
        i += 32;
        while (j < n && i >= n) {
          i -= n;
          ++j;
          i += j;
        }
      }
    }
    // forward solve of the right-hand sides, rows k+1..n-1
    const int m = n - k - 1;
    for (int e = lane; e < m * nrhs; e += 32) {
      const int c = e / m, i = k + 1 + (e - c * m);
      M[i * P + n + c] = fma_rn<T>(-M[i * P + k], M[k * P + n + c], M[i * P + n + c]);
    }
    __syncwarp();
  }
  __syncwarp();
  if (inf == 0) {
    // L^T x = y
    for (int k = n - 1; k >= 0; --k) {
      const T r = rcp[k];
      for (int c = lane; c < nrhs; c += 32) M[k * P + n + c] = M[k * P + n + c] * r;
      __syncwarp();
      for (int e = lane; e < k * nrhs; e += 32) {
        const int c = e / k, i = e - c * k;
        M[i * P + n + c] = fma_rn<T>(-M[k * P + i], M[k * P + n + c], M[i * P + n + c]);
      }
      __syncwarp();
    }
  }
  store_system<T>(A, B, M, n, nrhs, P, layout, true, inf != 0, lane);
  if (lane == 0) info[s] = inf;
}

}  // namespace

size_t lu_smem_bytes(int n, int nrhs, int elem_size) {
  const int P = odd_pitch(n + nrhs);
  return static_cast<size_t>(n) * P * elem_size + static_cast<size_t>(n) * elem_size +
         static_cast<size_t>(n) * sizeof(int);
}

size_t chol_smem_bytes(int n, int nrhs, int elem_size) {
  const int P = odd_pitch(n + nrhs);
  return static_cast<size_t>(n) * P * elem_size + static_cast<size_t>(n) * elem_size;
}

template <typename T>
cudaError_t launch_lu_smem(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                           int32_t* ipiv, int32_t* info, cudaStream_t stream) {
  if (batch > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const size_t bytes = lu_smem_bytes(n, nrhs, sizeof(T));
  cudaError_t e = cudaFuncSetAttribute(lu_smem_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  lu_smem_kernel<T><<<static_cast<unsigned>(batch), 32, bytes, stream>>>(n, nrhs, layout, batch,
                                                                         A, B, ipiv, info);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_chol_smem(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                             int32_t* info, cudaStream_t stream) {
  if (batch > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const size_t bytes = chol_smem_bytes(n, nrhs, sizeof(T));
  cudaError_t e = cudaFuncSetAttribute(chol_smem_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  chol_smem_kernel<T><<<static_cast<unsigned>(batch), 32, bytes, stream>>>(n, nrhs, layout,
                                                                           batch, A, B, info);
  return cudaGetLastError();
}

template cudaError_t launch_lu_smem<float>(int, int, int, int64_t, float*, float*, int32_t*,
                                           int32_t*, cudaStream_t);
template cudaError_t launch_lu_smem<double>(int, int, int, int64_t, double*, double*, int32_t*,
                                            int32_t*, cudaStream_t);
template cudaError_t launch_chol_smem<float>(int, int, int, int64_t, float*, float*, int32_t*,
                                             cudaStream_t);
template cudaError_t launch_chol_smem<double>(int, int, int, int64_t, double*, double*,
                                              int32_t*, cudaStream_t);

}  // namespace bsolve
