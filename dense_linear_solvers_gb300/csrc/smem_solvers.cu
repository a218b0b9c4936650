// Lower Cholesky for 32 < n <= 128, one warp per system, with the system resident in
// shared memory (n <= 32 runs the lockstep kernel of chol_sys.cu).
//
// The system is held as one n x P row-major tile M = [A | B] (P = n + nrhs rounded up to
// an odd number of elements, so that walking down a column touches distinct banks).
// Every step of the right-looking factorization spreads its trailing update over the
// 32 lanes element by element (a column-major walk of the trailing block), so that the
// warp's instructions stay busy however small the trailing block gets; this matters on
// a part whose FP64 pipe charges a whole warp instruction whatever its active lanes.
//
// Cholesky: right-looking lower factorization (cuSolverDx docs, "Cholesky
// Factorization": only the lower triangle is read and written), the forward solve
// folded in, then L^T x = y. Under the RUDA status contract of the _ex call (RUDA docs,
// "ruSOLVER: small-matrix kernel optimisation", unchanged failure contract) the whole
// matrix is loaded so that its symmetry can be checked: -1 a non-finite input, -2 an input
// that is not symmetric, -3 a non-finite result; failures return zeros.
// The arithmetic is the CPU oracle's, operation by operation.
#include "common.cuh"
#include "kernels.h"

namespace bsolve {
namespace {

__host__ __device__ inline int odd_pitch(int w) { return w | 1; }

// layouts: bit 0 the storage order of A, bit 1 that of B. Element e of the system lives at
// A[e * st] (st = 1: the systems one after another; otherwise the interleaved batched
// layout), likewise B.
template <typename T>
__device__ __forceinline__ void load_system(const T* __restrict__ A, const T* __restrict__ B,
                                            T* M, int n, int nrhs, int P, int layouts,
                                            bool lower_only, int lane, int64_t st) {
  if ((layouts & 1) == kRowMajor) {
    for (int i = 0; i < n; ++i) {
      const int jend = lower_only ? i + 1 : n;
      for (int j = lane; j < jend; j += 32) M[i * P + j] = A[(i * n + j) * st];
    }
  } else {
    for (int j = 0; j < n; ++j)
      for (int i = (lower_only ? j : 0) + lane; i < n; i += 32) M[i * P + j] = A[(j * n + i) * st];
  }
  if ((layouts >> 1) == kRowMajor) {
    for (int e = lane; e < n * nrhs; e += 32) {
      const int i = e / nrhs, c = e - i * nrhs;
      M[i * P + n + c] = B[e * st];
    }
  } else {
    for (int c = 0; c < nrhs; ++c)
      for (int i = lane; i < n; i += 32) M[i * P + n + c] = B[(c * n + i) * st];
  }
}

template <typename T>
__device__ __forceinline__ void store_system(T* __restrict__ A, T* __restrict__ B, const T* M,
                                             int n, int nrhs, int P, int layouts,
                                             bool lower_only, bool zero_x, int lane, int64_t st) {
  if ((layouts & 1) == kRowMajor) {
    for (int i = 0; i < n; ++i) {
      const int jend = lower_only ? i + 1 : n;
      for (int j = lane; j < jend; j += 32) A[(i * n + j) * st] = M[i * P + j];
    }
  } else {
    for (int j = 0; j < n; ++j)
      for (int i = (lower_only ? j : 0) + lane; i < n; i += 32) A[(j * n + i) * st] = M[i * P + j];
  }
  if ((layouts >> 1) == kRowMajor) {
    for (int e = lane; e < n * nrhs; e += 32) {
      const int i = e / nrhs, c = e - i * nrhs;
      B[e * st] = zero_x ? T(0) : M[i * P + n + c];
    }
  } else {
    for (int c = 0; c < nrhs; ++c)
      for (int i = lane; i < n; i += 32) B[(c * n + i) * st] = zero_x ? T(0) : M[i * P + n + c];
  }
}

// IL: the interleaved batched layout (element stride ilv); the plain instance has stride 1
template <typename T, bool IL>
__global__ void __launch_bounds__(32)
chol_smem_kernel(int n, int nrhs, int layouts, int64_t batch, T* __restrict__ A,
                 T* __restrict__ B, int32_t* __restrict__ info, int ruda, int64_t ilv_) {
  const int64_t ilv = IL ? ilv_ : 1;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x;
  const int64_t s = blockIdx.x;
  if (s >= batch) return;
  const int P = odd_pitch(n + nrhs);
  T* M = reinterpret_cast<T*>(smem_raw);
  T* rcp = M + n * P;

  const int64_t blk = IL ? s / ilv : s, sl = IL ? s - blk * ilv : 0;
  A += blk * ilv * n * n + sl;
  B += blk * ilv * n * nrhs + sl;
  // the RUDA status contract reads the whole matrix: its symmetry is checked
  load_system<T>(A, B, M, n, nrhs, P, layouts, !ruda, lane, ilv);
  __syncwarp();

  int inf = 0;
  if (ruda) {
    bool bad = false, asym = false;
    const int W = n + nrhs;
    for (int e = lane; e < n * W; e += 32) {
      const int i = e / W, j = e - i * W;
      const T v = M[i * P + j];
      bad = bad || !isfinite(v);
      if (j < i) asym = asym || !(v == M[j * P + i]);
    }
    if (__any_sync(0xFFFFFFFFu, bad)) inf = -1;
    else if (__any_sync(0xFFFFFFFFu, asym)) inf = -2;
  }
  for (int k = 0; k < n && inf == 0; ++k) {
    const T d = M[k * P + k];
    if (!(d > T(0))) {
      inf = k + 1;
      break;
    }
    const T l = sqrt_rn<T>(d);
    const T r = rcp_rn<T>(l);
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
  if (inf == 0 && nrhs > 0) {
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
  if (ruda) {
    // -3: a non-finite factor or solution after a sweep without a failing minor; a failed
    // system returns the factor's triangle and X as zeros
    if (inf == 0) {
      bool bad = false;
      for (int e = lane; e < n * (n + nrhs); e += 32) {
        const int i = e / (n + nrhs), j = e - i * (n + nrhs);
        if (j <= i || j >= n) bad = bad || !isfinite(M[i * P + j]);
      }
      if (__any_sync(0xFFFFFFFFu, bad)) inf = -3;
    }
    if (inf != 0) {
      for (int e = lane; e < n * n; e += 32) {
        const int i = e / n, j = e - i * n;
        if (j <= i) M[i * P + j] = T(0);
      }
    }
    __syncwarp();
  }
  store_system<T>(A, B, M, n, nrhs, P, layouts, true, inf != 0, lane, ilv);
  if (lane == 0) info[s] = inf;
}

}  // namespace

size_t chol_smem_bytes(int n, int nrhs, int elem_size) {
  const int P = odd_pitch(n + nrhs);
  return static_cast<size_t>(n) * P * elem_size + static_cast<size_t>(n) * elem_size;
}

template <typename T>
cudaError_t launch_chol_smem_ex(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                                int32_t* info, int ruda, cudaStream_t stream, int64_t ilv) {
  if (batch > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  if (ilv < 1) return cudaErrorInvalidValue;
  const size_t bytes = chol_smem_bytes(n, nrhs, sizeof(T));
  cudaError_t e = cudaFuncSetAttribute(
      ilv == 1 ? chol_smem_kernel<T, false> : chol_smem_kernel<T, true>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (ilv == 1)
    chol_smem_kernel<T, false><<<static_cast<unsigned>(batch), 32, bytes, stream>>>(
        n, nrhs, layout, batch, A, B, info, ruda, 1);
  else
    chol_smem_kernel<T, true><<<static_cast<unsigned>(batch), 32, bytes, stream>>>(
        n, nrhs, layout, batch, A, B, info, ruda, ilv);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_chol_smem(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                             int32_t* info, cudaStream_t stream) {
  return launch_chol_smem_ex<T>(layout, n, nrhs, batch, A, B, info, 0, stream, 1);
}

template cudaError_t launch_chol_smem_ex<float>(int, int, int, int64_t, float*, float*, int32_t*,
                                                int, cudaStream_t, int64_t);
template cudaError_t launch_chol_smem_ex<double>(int, int, int, int64_t, double*, double*,
                                                 int32_t*, int, cudaStream_t, int64_t);
template cudaError_t launch_chol_smem<float>(int, int, int, int64_t, float*, float*, int32_t*,
                                             cudaStream_t);
template cudaError_t launch_chol_smem<double>(int, int, int, int64_t, double*, double*,
                                              int32_t*, cudaStream_t);

}  // namespace bsolve
