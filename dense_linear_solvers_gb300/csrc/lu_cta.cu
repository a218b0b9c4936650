// LU with partial pivoting + solve for 32 < n <= 128: one system per block of four warps,
// the system resident in shared memory.
//
// The system is one n x P row-major tile M = [A | B] (P = n + nrhs rounded up to an
// odd number of elements: a walk down a column touches distinct banks). The right-
// looking factorization follows LAPACK's order with physical row interchanges (TDLS
// API, "solver_static.hpp File Reference", Detailed Description: physical and logical
// interchanges choose the same pivots and run the same operations):
//   phase 1 (one warp, during the previous step's update: look-ahead): the update of
//     column k, then its pivot search with integer magnitude keys and the lowest-row tie
//     rule, and the correctly rounded pivot reciprocal;
//   phase 2 (all warps): the interchange of rows k and p and the multipliers of column k;
//   phase 3 (the other warps): the rank-1 update of rows k+1.., columns k+2.. of [A | B]
//     (the forward solve L y = P b folded in), spread element by element over their
//     lanes so that lanes stay busy however small the trailing block gets.
// On this part a warp FP64 instruction is charged whatever its active lanes, so the
// lane count that does useful FP64 work is what sets the speed; four warps per system
// also give the SM enough warps to cover each system's serial pivot phase. The serial
// warp rotates with the step and the block, so the serial work of the blocks on an SM is
// spread over its four sub-partitions.
// Options of the _ex calls (run here for every n): TDLS threshold pivoting (the row in
// place stays when |a_kk| >= tau * m, m the magnitude the search found) and the RUDA
// status contract (-1 for a non-finite input before the sweep, -3 for a non-finite factor
// or solution after it, failed systems returned as zeros with pivots -1), and RUDA's
// scaling by the largest magnitude of the matrix (A divided by it before the sweep when it
// is finite and positive, U multiplied by it after, the back substitution on the restored
// U with its reciprocals recomputed).
// Back substitution runs by blocks of four rows: one warp solves the 4 x 4 diagonal block,
// then all warps apply its four columns to every row above, each element taking the four
// updates in decreasing column order -- the oracle's order, so the arithmetic is the
// CPU oracle's, operation by operation.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace bsolve {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kBlk = 4;  // rows per back-substitution block

__host__ __device__ inline int odd_pitch(int w) { return w | 1; }

// IL: the interleaved batched layout (element stride ilv); the plain instance has stride 1
template <typename T, bool IL>
__global__ void __launch_bounds__(kThreads)
lu_cta_kernel(int n, int nrhs, int layout, int64_t batch, T* __restrict__ A,
              T* __restrict__ B, int32_t* __restrict__ ipiv, int32_t* __restrict__ info,
              T tau, int ruda, int64_t ilv_, int scale) {
  const int64_t ilv = IL ? ilv_ : 1;
  using Key = typename Traits<T>::Key;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int64_t s = blockIdx.x;
  if (s >= batch) return;
  const int W = n + nrhs;
  const int P = odd_pitch(W);
  T* const M = reinterpret_cast<T*>(smem_raw);
  T* const rcp = M + n * P;
  int* const piv = reinterpret_cast<int*>(rcp + n);
  __shared__ int s_info;
  __shared__ Key s_max;
  __shared__ int s_p;      // pivot row of the step being prepared
  __shared__ T s_pv, s_akk;

  // element e of the system at A[e * ilv] (ilv = 1: the systems one after another;
  // otherwise the interleaved batched layout, systems in blocks of ilv), likewise B, ipiv
  const int64_t blk = IL ? s / ilv : s, sl = IL ? s - blk * ilv : 0;
  A += blk * ilv * n * n + sl;
  B += blk * ilv * n * nrhs + sl;
  ipiv += blk * ilv * n + sl;
  // asynchronous element copies: every load of the system is in flight at once
  if (layout == kRowMajor) {
    for (int e = tid; e < n * n; e += kThreads) {
      const int i = e / n, j = e - i * n;
      cp_async_elem<T>(M + i * P + j, A + e * ilv);
    }
    for (int e = tid; e < n * nrhs; e += kThreads) {
      const int i = e / nrhs, c = e - i * nrhs;
      cp_async_elem<T>(M + i * P + n + c, B + e * ilv);
    }
  } else {
    for (int e = tid; e < n * n; e += kThreads) {
      const int j = e / n, i = e - j * n;
      cp_async_elem<T>(M + i * P + j, A + e * ilv);
    }
    for (int e = tid; e < n * nrhs; e += kThreads) {
      const int c = e / n, i = e - c * n;
      cp_async_elem<T>(M + i * P + n + c, B + e * ilv);
    }
  }
  if (tid == 0) {
    s_info = 0;
    s_max = 0;
  }
  cp_async_wait_all();
  __syncthreads();

  // RUDA status contract: a non-finite input fails the system with -1 before the sweep
  if (ruda) {
    int bad = 0;
    for (int e = tid; e < n * W; e += kThreads) {
      const int i = e / W, j = e - i * W;
      bad |= !isfinite(M[i * P + j]);
    }
    if (__syncthreads_or(bad)) {
      for (int e = tid; e < n * n; e += kThreads) A[e * ilv] = T(0);
      for (int e = tid; e < n * nrhs; e += kThreads) B[e * ilv] = T(0);
      for (int k = tid; k < n; k += kThreads) ipiv[k * ilv] = -1;
      if (tid == 0) info[s] = -1;
      return;
    }
  }

  // RUDA scaling: m = max |a_ij| (as magnitude bits: their order is the values'); a
  // non-finite entry leaves the system unscaled
  T msc = T(0);
  if (scale) {
    Key mk = 0;
    int nonfin = 0;
    for (int e = tid; e < n * n; e += kThreads) {
      const int i = e / n, j = e - i * n;
      const Key kb = Traits<T>::mag_bits(M[i * P + j]);
      nonfin |= kb >= Traits<T>::kInfBits;
      mk = kb > mk ? kb : mk;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const Key o = shfl_xor_key(mk, off, 32);
      mk = o > mk ? o : mk;
    }
    if (lane == 0) atomicMax(&s_max, mk);
    nonfin = __syncthreads_or(nonfin);
    if (!nonfin && s_max > 0) {
      msc = pivot_from_key<T>(s_max + 1, 0u);   // a key is the magnitude bits + 1
      for (int e = tid; e < n * n; e += kThreads) {
        const int i = e / n, j = e - i * n;
        M[i * P + j] = M[i * P + j] / msc;
      }
    }
    __syncthreads();
  }

  // The pivot search of column kk (rows kk..n-1) on the calling warp; it moves no data:
  // the pivot row, the pivot and the old a_kk go to shared scalars, ipiv, info and the
  // pivot reciprocal to their arrays. A lane keeps its first maximum; the lowest row wins
  // a tie.
  auto search = [&](int kk) {
    Key best = 0;
    int bi = 0x7FFFFFFF;
    for (int i = kk + lane; i < n; i += 32) {
      const Key key = pivot_key<T>(M[i * P + kk], i == kk);
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
    int p = bi;
    Key pkey = best;
    const T akk = M[kk * P + kk];
    if (p != kk && tau < T(1)) {
      // threshold pivoting: the row in place stays when |a_kk| >= tau * m, m the
      // magnitude the search found (not a NaN: a NaN in place would have won)
      if (fabs(akk) >= tau * pivot_from_key<T>(best, 0u)) {
        p = kk;
        pkey = pivot_key<T>(akk, true);
      }
    }
    const bool ok = pivot_ok<T>(pkey);
    if (lane == 0) {
      const T pv = M[p * P + kk];
      piv[kk] = p + 1;
      if (!ok && s_info == 0) s_info = kk + 1;
      rcp[kk] = ok ? rcp_rn<T>(pv) : T(1);
      s_p = p;
      s_pv = pv;
      s_akk = akk;
    }
  };
  // All threads: rows kk and p exchanged over every column but kk, and column kk below the
  // diagonal scaled by the pivot reciprocal, its entries at kk and p taken from the
  // scalars the search saved (so no thread reads what another writes).
  auto swap_scale = [&](int kk) {
    const int p = s_p;
    const T r = rcp[kk];
    if (p != kk) {
      for (int j = tid; j < W; j += kThreads) {
        if (j == kk) continue;
        const T t = M[kk * P + j];
        M[kk * P + j] = M[p * P + j];
        M[p * P + j] = t;
      }
    }
    for (int i = kk + tid; i < n; i += kThreads) {
      if (i == kk)
        M[i * P + kk] = s_pv;
      else if (i == p)
        M[i * P + kk] = s_akk * r;
      else
        M[i * P + kk] = M[i * P + kk] * r;
    }
  };
  // the search of column kk runs on a warp that rotates with the column and the block:
  // warp w runs on SM sub-partition w % 4, and a fixed warp would put every block's
  // serial work on one sub-partition
  auto chain = [&](int kk) { return (static_cast<int>(blockIdx.x) + kk) & (kWarps - 1); };

  if (warp == chain(0)) search(0);
  __syncthreads();
  swap_scale(0);
  __syncthreads();
  for (int k = 0; k < n; ++k) {
    // rank-1 update of rows k+1..n-1, columns k+1..W-1 (look-ahead: the chain warp of
    // column k+1 updates that column and searches its pivot while the other warps update
    // the columns after it; the exchange and scaling of step k+1 follow the barrier)
    const int m = n - k - 1;
    const bool ahead = k + 1 < n;
    const int cw = ahead ? chain(k + 1) : -1;
    if (warp == cw) {
      for (int i = k + 1 + lane; i < n; i += 32)
        M[i * P + k + 1] = fma_rn<T>(-M[i * P + k], M[k * P + k + 1], M[i * P + k + 1]);
      __syncwarp();
      search(k + 1);
    } else if (m > 0) {
      const int j0 = ahead ? k + 2 : k + 1;
      const int w = W - j0;
      const int nth = ahead ? kThreads - 32 : kThreads;
      const int t = (ahead && warp > cw) ? tid - 32 : tid;
      const int total = m * w;
      const int dq = nth / m, dr = nth - dq * m;
      int ii = t % m, jj = t / m;
      for (int e = t; e < total; e += nth) {
        const int i = k + 1 + ii, j = j0 + jj;
        M[i * P + j] = fma_rn<T>(-M[i * P + k], M[k * P + j], M[i * P + j]);
        ii += dr;
        jj += dq;
        if (ii >= m) {
          ii -= m;
          ++jj;
        }
      }
    }
    __syncthreads();
    if (ahead) {
      swap_scale(k + 1);
      __syncthreads();
    }
  }

  // RUDA scaling: U's scale restored, and the reciprocals of its diagonal recomputed for
  // the back substitution (a pivot below the smallest normal number gets 1)
  if (msc > T(0)) {
    for (int e = tid; e < n * n; e += kThreads) {
      const int i = e / n, j = e - i * n;
      if (j >= i) M[i * P + j] = M[i * P + j] * msc;
    }
    __syncthreads();
    const T fl = sizeof(T) == 4 ? T(FLT_MIN) : T(DBL_MIN);
    for (int k = tid; k < n; k += kThreads) {
      const T u = M[k * P + k];
      rcp[k] = fabs(u) >= fl ? rcp_rn<T>(u) : T(1);
    }
    __syncthreads();
  }

  // U x = y by blocks of kBlk rows, from the last block (nothing to do without B)
  const int nblk = nrhs > 0 ? (n + kBlk - 1) / kBlk : 0;
  for (int cb = nblk - 1; cb >= 0; --cb) {
    const int lo = cb * kBlk, hi = min(n, lo + kBlk);
    if (warp == ((static_cast<int>(blockIdx.x) + cb) & (kWarps - 1))) {
      for (int i = hi - 1; i >= lo; --i) {
        const T r = rcp[i];
        for (int c = lane; c < nrhs; c += 32) M[i * P + n + c] = M[i * P + n + c] * r;
        __syncwarp();
        const int cnt = (i - lo) * nrhs;
        for (int e = lane; e < cnt; e += 32) {
          const int c = e / (i - lo), i2 = lo + (e - c * (i - lo));
          M[i2 * P + n + c] = fma_rn<T>(-M[i2 * P + i], M[i * P + n + c], M[i2 * P + n + c]);
        }
        __syncwarp();
      }
    }
    __syncthreads();
    // the block's columns applied to every row above it, decreasing column order
    const int cnt = lo * nrhs;
    for (int e = tid; e < cnt; e += kThreads) {
      const int c = e / lo, i2 = e - c * lo;
      T y = M[i2 * P + n + c];
      for (int i = hi - 1; i >= lo; --i) y = fma_rn<T>(-M[i2 * P + i], M[i * P + n + c], y);
      M[i2 * P + n + c] = y;
    }
    __syncthreads();
  }

  // RUDA status contract: a non-finite factor or solution after a sweep without a failing
  // pivot is -3; a failed system returns zeros and pivots -1
  int status = s_info;
  if (ruda) {
    int bad = 0;
    if (status == 0) {
      for (int e = tid; e < n * W; e += kThreads) {
        const int i = e / W, j = e - i * W;
        bad |= !isfinite(M[i * P + j]);
      }
    }
    if (__syncthreads_or(bad)) status = -3;
  }
  const bool zero_all = ruda && status != 0;
  const bool zero_x = status != 0;
  if (layout == kRowMajor) {
    for (int e = tid; e < n * n; e += kThreads) {
      const int i = e / n, j = e - i * n;
      A[e * ilv] = zero_all ? T(0) : M[i * P + j];
    }
    for (int e = tid; e < n * nrhs; e += kThreads) {
      const int i = e / nrhs, c = e - i * nrhs;
      B[e * ilv] = zero_x ? T(0) : M[i * P + n + c];
    }
  } else {
    for (int e = tid; e < n * n; e += kThreads) {
      const int j = e / n, i = e - j * n;
      A[e * ilv] = zero_all ? T(0) : M[i * P + j];
    }
    for (int e = tid; e < n * nrhs; e += kThreads) {
      const int c = e / n, i = e - c * n;
      B[e * ilv] = zero_x ? T(0) : M[i * P + n + c];
    }
  }
  for (int k = tid; k < n; k += kThreads) ipiv[k * ilv] = zero_all ? -1 : piv[k];
  if (tid == 0) info[s] = status;
}

}  // namespace

size_t lu_cta_bytes(int n, int nrhs, int elem_size) {
  const int P = odd_pitch(n + nrhs);
  return static_cast<size_t>(n) * P * elem_size + static_cast<size_t>(n) * elem_size +
         static_cast<size_t>(n) * sizeof(int);
}

template <typename T>
cudaError_t launch_lu_smem_ex(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                              int32_t* ipiv, int32_t* info, double tau, int ruda,
                              cudaStream_t stream, int64_t ilv, int scale) {
  if (ilv < 1) return cudaErrorInvalidValue;
  if (batch > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const size_t bytes = lu_cta_bytes(n, nrhs, sizeof(T));
  cudaError_t e = cudaFuncSetAttribute(
      ilv == 1 ? lu_cta_kernel<T, false> : lu_cta_kernel<T, true>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (ilv == 1)
    lu_cta_kernel<T, false><<<static_cast<unsigned>(batch), kThreads, bytes, stream>>>(
        n, nrhs, layout, batch, A, B, ipiv, info, static_cast<T>(tau), ruda, 1, scale);
  else
    lu_cta_kernel<T, true><<<static_cast<unsigned>(batch), kThreads, bytes, stream>>>(
        n, nrhs, layout, batch, A, B, ipiv, info, static_cast<T>(tau), ruda, ilv, scale);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_lu_smem(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                           int32_t* ipiv, int32_t* info, cudaStream_t stream) {
  return launch_lu_smem_ex<T>(layout, n, nrhs, batch, A, B, ipiv, info, 1.0, 0, stream, 1, 0);
}

template cudaError_t launch_lu_smem<float>(int, int, int, int64_t, float*, float*, int32_t*,
                                           int32_t*, cudaStream_t);
template cudaError_t launch_lu_smem<double>(int, int, int, int64_t, double*, double*, int32_t*,
                                            int32_t*, cudaStream_t);
template cudaError_t launch_lu_smem_ex<float>(int, int, int, int64_t, float*, float*, int32_t*,
                                              int32_t*, double, int, cudaStream_t, int64_t, int);
template cudaError_t launch_lu_smem_ex<double>(int, int, int, int64_t, double*, double*,
                                               int32_t*, int32_t*, double, int, cudaStream_t,
                                               int64_t, int);

}  // namespace bsolve
