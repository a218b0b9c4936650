// Lower Cholesky + solve for n <= 32: sixteen systems per block, computed in lockstep
// with one system per lane.
//
// On a part whose FP64 pipe runs at 1/64 of the FP32 lane rate and charges a warp
// instruction whatever its active lanes, the per-column scalar chain of Cholesky (a
// square root and a reciprocal, several FP64 instructions each) is ruinous when a warp
// works on one system: it costs as much as a whole column's update. Here every warp
// instruction works on the same element of sixteen systems (lane l -> system l % 16,
// half-warp l / 16 -> one of two element slots), so the scalar chain of sixteen systems
// costs one instruction sequence, and the trailing update runs as many elements per
// instruction as there are lanes, with no idle lanes however small the trailing
// triangle gets.
//
// Each system lives in shared memory as a packed lower triangle (row i at i(i+1)/2)
// followed by its right-hand sides (row i at tri + i*nrhs). The per-system stride is an
// odd number of elements, so the sixteen lanes that touch the same element of sixteen
// systems hit sixteen different banks.
//
// The factorization is right-looking (cuSolverDx docs, "Cholesky Factorization": only
// the lower triangle is read and replaced by L; info = the smallest leading minor that
// is not positive definite), with the forward solve folded into it; then L^T x = y.
// Per column k: scale column k (all warps), barrier, then the trailing update on all warps
// but one, the chain warp of column k+1, which updates a_{k+1,k+1} only and takes column
// k+1's square root and reciprocal at once (look-ahead: the serial chain overlaps the
// update and needs no barrier of its own), barrier.
// The arithmetic is the CPU oracle's, operation by operation. A system whose minor
// fails keeps computing (no branch depends on the data) and returns X = 0.
#include "common.cuh"
#include "kernels.h"

namespace bsolve {
namespace {

constexpr int kSys = 16;      // systems per block
constexpr int kWarps = 16;    // warps per block (3 blocks per SM by shared memory: 48 warps)
constexpr int kSlots = kWarps * 2;
constexpr int kMaxN = 32;

__host__ __device__ inline int tri(int i) { return i * (i + 1) / 2; }

__host__ __device__ inline int sys_stride(int n, int nrhs) { return (tri(n) + n * nrhs) | 1; }

// IL: the interleaved batched layout (element stride ilv); the plain instance has stride 1
template <typename T, bool IL>
__global__ void __launch_bounds__(kWarps * 32)
chol_sys_kernel(int n, int nrhs, int layouts, int64_t batch, T* __restrict__ A,
                T* __restrict__ B, int32_t* __restrict__ info, int64_t ilv_) {
  const int64_t ilv = IL ? ilv_ : 1;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int alay = layouts & 1, blay = layouts >> 1;   // storage orders of A and of B
  const int D = sys_stride(n, nrhs);
  const int TRI = tri(n);
  T* const M = reinterpret_cast<T*>(smem_raw);     // kSys systems, stride D
  T* const rr = M + kSys * D;                       // [kMaxN][kSys] reciprocals
  int* const sinfo = reinterpret_cast<int*>(rr + kSys * kMaxN);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int s = lane & (kSys - 1);                  // system of this lane
  const int slot = warp * 2 + (lane >> 4);          // element slot of this lane
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kSys;
  T* const Ms = M + s * D;                          // this lane's system
  T* const Ys = Ms + TRI;                           // its right-hand sides, [i][c]

  // Element e of system sys at As[e * ilv]: ilv = 1, the systems one after another (each
  // warp copies whole systems, its lanes walking the rows of a column); otherwise the
  // interleaved batched layout, where the block's sixteen systems hold each element side by
  // side, so each half-warp copies one element of all sixteen (128 contiguous bytes in
  // FP64 when they lie in one block of ilv). Asynchronous element copies keep every load
  // of the block in flight at once.
  auto sys_base = [&](int64_t sys, T* P, int size) {
    const int64_t blk = IL ? sys / ilv : sys, sl = IL ? sys - blk * ilv : 0;
    return P + blk * ilv * size + sl;
  };
  if constexpr (IL) {
    // thread -> system tid % 16 and element slot tid / 16 of each pass (kSlots per pass);
    // the lower triangle walked row by row (row i: columns 0..i), then B by rows
    const int q = tid % kSys, e0 = tid / kSys;
    const int64_t sys = s0 + q;
    T* const Mq = M + q * D;
    if (sys < batch) {
      const T* As = sys_base(sys, A, n * n);
      const T* Bs = sys_base(sys, B, n * nrhs);
      int i = 0, j = e0;
      while (j > i) {
        j -= i + 1;
        ++i;
      }
      for (int t = e0; t < TRI; t += kSlots) {
        cp_async_elem<T>(Mq + t, As + (alay == kColMajor ? j * n + i : i * n + j) * ilv);
        j += kSlots;
        while (j > i) {
          j -= i + 1;
          ++i;
        }
      }
      for (int f = e0; f < n * nrhs; f += kSlots) {
        const int i2 = f / nrhs, c = f - i2 * nrhs;
        cp_async_elem<T>(Mq + TRI + f,
                         Bs + (blay == kColMajor ? c * n + i2 : i2 * nrhs + c) * ilv);
      }
    } else {
      // a system past the end of the batch: an identity keeps its lanes finite (each
      // element written once, by the thread that owns it)
      int i = 0, j = e0;
      while (j > i) {
        j -= i + 1;
        ++i;
      }
      for (int t = e0; t < TRI; t += kSlots) {
        Mq[t] = i == j ? T(1) : T(0);
        j += kSlots;
        while (j > i) {
          j -= i + 1;
          ++i;
        }
      }
      for (int e = TRI + e0; e < D; e += kSlots) Mq[e] = T(0);
    }
    if (e0 == 0) sinfo[q] = 0;
  } else {
    for (int q = warp; q < kSys; q += kWarps) {
      const int64_t sys = s0 + q;
      T* const Mq = M + q * D;
      if (sys < batch) {
        const T* As = sys_base(sys, A, n * n);
        const T* Bs = sys_base(sys, B, n * nrhs);
        for (int j = 0; j < n; ++j)
          for (int i = j + lane; i < n; i += 32)
            cp_async_elem<T>(Mq + tri(i) + j,
                             As + (alay == kColMajor ? j * n + i : i * n + j) * ilv);
        for (int c = 0; c < nrhs; ++c)
          for (int i = lane; i < n; i += 32)
            cp_async_elem<T>(Mq + TRI + i * nrhs + c,
                             Bs + (blay == kColMajor ? c * n + i : i * nrhs + c) * ilv);
      } else {
        // a system past the end of the batch: an identity keeps its lanes finite
        for (int e = lane; e < D; e += 32) Mq[e] = T(0);
        __syncwarp();
        for (int i = lane; i < n; i += 32) Mq[tri(i) + i] = T(1);
      }
      if (lane == 0) sinfo[q] = 0;
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // A: the pivot of column kk, one lane per system (lanes 0..15 of the chain warp): the
  //    square root and its reciprocal; the first failing minor sets info
  auto pivot = [&](int kk) {
    const T d = Ms[tri(kk) + kk];
    if (!(d > T(0)) && sinfo[s] == 0) sinfo[s] = kk + 1;
    const T l = sqrt_rn<T>(d);
    Ms[tri(kk) + kk] = l;
    rr[kk * kSys + s] = rcp_rn<T>(l);
  };
  // the chain warp of column kk rotates with the column and the block: warp w runs on SM
  // sub-partition w % 4, so a fixed warp would put every block's chain on one FP64 pipe
  auto chain_warp = [&](int kk) { return (static_cast<int>(blockIdx.x) + kk) & (kWarps - 1); };
  if (warp == chain_warp(0) && lane < kSys) pivot(0);
  __syncthreads();

  for (int k = 0; k < n; ++k) {
    // B: scale column k below the diagonal, and y_k
    {
      const int m = n - 1 - k;
      const T r = rr[k * kSys + s];
      for (int e = slot; e < m + nrhs; e += kSlots) {
        if (e < m) {
          const int i = k + 1 + e;
          Ms[tri(i) + k] = Ms[tri(i) + k] * r;
        } else {
          const int c = e - m;
          Ys[k * nrhs + c] = Ys[k * nrhs + c] * r;
        }
      }
    }
    __syncthreads();
    // C: trailing lower triangle (row by row: row i holds columns k+1..i), then the
    //    forward solve of rows k+1..n-1. Element 0, a_{k+1,k+1}, belongs to the chain
    //    warp of column k+1, which then takes that column's pivot (A) at once and does
    //    nothing else, so the serial chain overlaps the rest of the update (spread over
    //    the other warps' slots) and needs no barrier of its own.
    {
      const int m = n - 1 - k;
      const int T_k = m * (m + 1) / 2;
      const int cw = chain_warp(k + 1);
      if (warp == cw) {
        if (m > 0 && lane < kSys) {
          const int t1 = tri(k + 1);
          Ms[t1 + k + 1] = fma_rn<T>(-Ms[t1 + k], Ms[t1 + k], Ms[t1 + k + 1]);
          pivot(k + 1);
        }
      } else {
        constexpr int kOther = kSlots - 2;             // the other warps' slots
        const int vs = slot < 2 * cw ? slot : slot - 2;
        int i = k + 1, j = k + 2 + vs;                 // element 1 + vs
        while (i < n && j > i) {
          j -= i - k;
          ++i;
        }
        for (int e = 1 + vs; e < T_k; e += kOther) {
          const int ti = tri(i);
          Ms[ti + j] = fma_rn<T>(-Ms[ti + k], Ms[tri(j) + k], Ms[ti + j]);
          j += kOther;
          while (i < n && j > i) {
            j -= i - k;
            ++i;
          }
        }
        for (int f = vs; f < m * nrhs; f += kOther) {
          const int ii = k + 1 + f / nrhs, c = f - (f / nrhs) * nrhs;
          Ys[ii * nrhs + c] = fma_rn<T>(-Ms[tri(ii) + k], Ys[k * nrhs + c], Ys[ii * nrhs + c]);
        }
      }
    }
    __syncthreads();
  }

  // L^T x = y, from the last row. x_k = y_k * r_k is taken by whichever thread gives
  // y_k its last update (in step k+1), so each step needs a single barrier.
  for (int c = slot; c < nrhs; c += kSlots) Ys[(n - 1) * nrhs + c] *= rr[(n - 1) * kSys + s];
  __syncthreads();
  for (int k = nrhs > 0 ? n - 1 : 0; k >= 1; --k) {   // nothing to do without B
    const int tk = tri(k);
    const T rkm1 = rr[(k - 1) * kSys + s];
    for (int e = slot; e < k * nrhs; e += kSlots) {
      const int i = e / nrhs, c = e - i * nrhs;
      T y = fma_rn<T>(-Ms[tk + i], Ys[k * nrhs + c], Ys[i * nrhs + c]);
      if (i == k - 1) y = y * rkm1;
      Ys[i * nrhs + c] = y;
    }
    __syncthreads();
  }

  // store: the lower triangle, X (zero for a failed system), info; the same thread to
  // element maps as the load
  if constexpr (IL) {
    const int q = tid % kSys, e0 = tid / kSys;
    const int64_t sys = s0 + q;
    if (sys < batch) {
      const T* const Mq = M + q * D;
      T* As = sys_base(sys, A, n * n);
      T* Bs = sys_base(sys, B, n * nrhs);
      const bool failed = sinfo[q] != 0;
      int i = 0, j = e0;
      while (j > i) {
        j -= i + 1;
        ++i;
      }
      for (int t = e0; t < TRI; t += kSlots) {
        As[(alay == kColMajor ? j * n + i : i * n + j) * ilv] = Mq[t];
        j += kSlots;
        while (j > i) {
          j -= i + 1;
          ++i;
        }
      }
      for (int f = e0; f < n * nrhs; f += kSlots) {
        const int i2 = f / nrhs, c = f - i2 * nrhs;
        Bs[(blay == kColMajor ? c * n + i2 : i2 * nrhs + c) * ilv] = failed ? T(0) : Mq[TRI + f];
      }
      if (e0 == 0) info[sys] = sinfo[q];
    }
  } else {
    for (int q = warp; q < kSys; q += kWarps) {
      const int64_t sys = s0 + q;
      if (sys >= batch) continue;
      const T* const Mq = M + q * D;
      T* As = sys_base(sys, A, n * n);
      T* Bs = sys_base(sys, B, n * nrhs);
      const bool failed = sinfo[q] != 0;
      for (int j = 0; j < n; ++j)
        for (int i = j + lane; i < n; i += 32)
          As[(alay == kColMajor ? j * n + i : i * n + j) * ilv] = Mq[tri(i) + j];
      for (int c = 0; c < nrhs; ++c)
        for (int i = lane; i < n; i += 32)
          Bs[(blay == kColMajor ? c * n + i : i * nrhs + c) * ilv] =
              failed ? T(0) : Mq[TRI + i * nrhs + c];
      if (lane == 0) info[sys] = sinfo[q];
    }
  }
}

}  // namespace

size_t chol_sys_bytes(int n, int nrhs, int elem_size) {
  return static_cast<size_t>(kSys) * sys_stride(n, nrhs) * elem_size +
         static_cast<size_t>(kSys) * kMaxN * elem_size + kSys * sizeof(int);
}

template <typename T>
cudaError_t launch_chol_sys(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                            int32_t* info, cudaStream_t stream, int64_t ilv) {
  if (n > kMaxN || ilv < 1) return cudaErrorInvalidValue;
  const int64_t blocks = (batch + kSys - 1) / kSys;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const size_t bytes = chol_sys_bytes(n, nrhs, sizeof(T));
  cudaError_t e = cudaFuncSetAttribute(
      ilv == 1 ? chol_sys_kernel<T, false> : chol_sys_kernel<T, true>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (ilv == 1)
    chol_sys_kernel<T, false><<<static_cast<unsigned>(blocks), kWarps * 32, bytes, stream>>>(
        n, nrhs, layout, batch, A, B, info, 1);
  else
    chol_sys_kernel<T, true><<<static_cast<unsigned>(blocks), kWarps * 32, bytes, stream>>>(
        n, nrhs, layout, batch, A, B, info, ilv);
  return cudaGetLastError();
}

template cudaError_t launch_chol_sys<float>(int, int, int, int64_t, float*, float*, int32_t*,
                                            cudaStream_t, int64_t);
template cudaError_t launch_chol_sys<double>(int, int, int, int64_t, double*, double*,
                                             int32_t*, cudaStream_t, int64_t);

}  // namespace bsolve
