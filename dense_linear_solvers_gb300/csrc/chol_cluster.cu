// Cholesky for 128 < n <= 256: the lower triangle of one system spread over the shared
// memory of a thread-block cluster of four CTAs (cuSolverDx docs, "Cholesky
// Factorization", the cluster / distributed-shared-memory tiling for orders beyond one
// CTA), and the solve with the stored factor, one CTA per system.
//
// Factor: the lower triangle in 32 x 32 tiles; tile t = i(i+1)/2 + j of tile row i and
// tile column j <= i lives in CTA t % 4, slot t / 4. Right-looking by tile columns k:
//   1. the owner of tile (k,k) factors it with one warp (lane r holds row r in registers;
//      column c: l_cc = sqrt(a_cc), r_c = 1/l_cc, l_rc = a_rc r_c, then
//      a_rj -= l_rc l_jc for c < j <= r, the multipliers broadcast by shuffles);
//   2. cluster barrier; every CTA copies L_kk and the reciprocals out of the owner's
//      shared memory (distributed shared memory loads) and scales its own tiles (i,k),
//      i > k, one thread per row, column by column (l_rc = a_rc r_c, then
//      a_rj -= l_rc l_jc for the tile's later columns);
//   3. cluster barrier; every CTA copies the panel tiles (i,k) of the other CTAs into a
//      local buffer and applies the 32 updates of the panel to each of its trailing tiles
//      (i,j), k < j <= i, element (r, c) taking a_rc -= l_rK l_cK in increasing K.
// Every element thus takes the oracle's right-looking updates in increasing column order,
// each one fused multiply-add, so the factor is the oracle's bit for bit. Orders that are
// not a multiple of 32 are padded with identity rows and columns at the end: they come
// after every real column and never update a real entry. Remote tiles are read with
// distributed-shared-memory loads only (no TMA multicast); the code serves one GPU.
// After a failing minor (the first !(d > 0)) the sweep runs on to the end; info is the
// first failure and the factor from there on is unspecified.
//
// Solve (potrs, n > 128): one CTA per system, the right-hand sides eight columns at a
// time in shared memory, the factor staged from global memory a tile column at a time:
// forward y = L^{-1} b (the diagonal block by one warp, y_K = b_K (1/l_KK) broadcast by
// shuffles, then each row below takes its 32 updates in increasing K), backward
// x = L^{-T} y (each row of the block first takes the updates of the rows below in
// decreasing K, then the diagonal block from the last row up). The oracle's potrs order.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace bsolve {
namespace {

constexpr int TS = 32;          // tile order
constexpr int TP = TS + 1;      // tile pitch (odd: walks down a column hit distinct banks)
constexpr int CL = 4;           // CTAs per cluster
constexpr int kMaxT = 8;        // tiles per dimension: n <= 256
constexpr int kMaxTiles = kMaxT * (kMaxT + 1) / 2;
constexpr int kMaxSlots = (kMaxTiles + CL - 1) / CL;
constexpr int kThreads = 256;
constexpr int kTile = TS * TP;  // elements of one staged tile

__host__ __device__ constexpr int tile_index(int i, int j) { return i * (i + 1) / 2 + j; }

__device__ __forceinline__ int64_t gidx(int layout, int n, int r, int c) {
  return layout == kRowMajor ? static_cast<int64_t>(r) * n + c : static_cast<int64_t>(c) * n + r;
}
// element (r, c) of the n x nrhs right-hand sides
__device__ __forceinline__ int64_t bidx(int layout, int n, int nrhs, int r, int c) {
  return layout == kRowMajor ? static_cast<int64_t>(r) * nrhs + c
                             : static_cast<int64_t>(c) * n + r;
}

template <typename T>
size_t cluster_smem_bytes() {
  // owned tiles, the staged panel (tile rows 0..kMaxT-1, row k holding L_kk), the diagonal
  // reciprocals (own and staged), the first failure
  return static_cast<size_t>(kMaxSlots + kMaxT) * kTile * sizeof(T) + 2 * TS * sizeof(T) + 16;
}

// Factor the diagonal tile at `a` (pitch TP) with one warp; lane r owns row r. k is the
// tile column (for the global index of a failing minor), n the order.
template <typename T>
__device__ void potrf_tile(T* a, T* rc, int k, int n, int* fail) {
  const int r = threadIdx.x & 31;
  T v[TS];
#pragma unroll
  for (int j = 0; j < TS; ++j) v[j] = a[r * TP + j];
  int first = 0x7FFFFFFF;
#pragma unroll
  for (int c = 0; c < TS; ++c) {
    const T d = __shfl_sync(0xFFFFFFFFu, v[c], c);
    if (!(d > T(0)) && k * TS + c < n && first == 0x7FFFFFFF) first = k * TS + c + 1;
    const T l = sqrt_rn<T>(d);
    const T rr = rcp_rn<T>(l);
    if (r == c) v[c] = l;
    if (r > c) v[c] = v[c] * rr;
    if (r == 0) rc[c] = rr;
#pragma unroll
    for (int j = c + 1; j < TS; ++j) {
      const T ljc = __shfl_sync(0xFFFFFFFFu, v[c], j);
      if (r >= j) v[j] = fma_rn<T>(-v[c], ljc, v[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < TS; ++j) a[r * TP + j] = v[j];
  if (r == 0 && first < *fail) *fail = first;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
chol_cluster_kernel(int n, int alay, int64_t batch, T* __restrict__ A, int32_t* __restrict__ info) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int64_t s = blockIdx.x / CL;
  extern __shared__ __align__(16) unsigned char raw[];
  T* const tiles = reinterpret_cast<T*>(raw);
  T* const panel = tiles + kMaxSlots * kTile;
  T* const rc = panel + kMaxT * kTile;      // reciprocals of the tile this CTA factored
  T* const rcs = rc + TS;                  // staged reciprocals of L_kk
  int* const fail = reinterpret_cast<int*>(rcs + TS);
  const int tid = threadIdx.x;
  const int nt = (n + TS - 1) / TS;
  const int ntiles = nt * (nt + 1) / 2;
  T* const As = A + s * static_cast<int64_t>(n) * n;

  // the owned tiles of the lower triangle (the strict upper triangle is never read);
  // phantom rows and columns past n: identity
  for (int t = rank; t < ntiles; t += CL) {
    int i = 0;
    while (tile_index(i + 1, 0) <= t) ++i;
    const int j = t - tile_index(i, 0);
    T* dst = tiles + (t / CL) * kTile;
    for (int e = tid; e < TS * TS; e += kThreads) {
      // consecutive threads walk the contiguous direction of the storage order
      const int r = alay == kRowMajor ? e / TS : e % TS;
      const int c = alay == kRowMajor ? e % TS : e / TS;
      const int I = i * TS + r, J = j * TS + c;
      T v;
      if (I < n && J < n) v = I >= J ? As[gidx(alay, n, I, J)] : T(0);
      else v = I == J ? T(1) : T(0);
      dst[r * TP + c] = v;
    }
  }
  if (tid == 0) *fail = 0x7FFFFFFF;
  __syncthreads();

  for (int k = 0; k < nt; ++k) {
    const int tkk = tile_index(k, k);
    if (tkk % CL == rank && tid < 32) potrf_tile<T>(tiles + (tkk / CL) * kTile, rc, k, n, fail);
    cluster.sync();
    // L_kk and its reciprocals from the owner
    {
      const T* src = cluster.map_shared_rank(tiles + (tkk / CL) * kTile, tkk % CL);
      T* dst = panel + k * kTile;
      for (int e = tid; e < kTile; e += kThreads) dst[e] = src[e];
      const T* rsrc = cluster.map_shared_rank(rc, tkk % CL);
      if (tid < TS) rcs[tid] = rsrc[tid];
    }
    __syncthreads();
    // the owned panel tiles (i,k), i > k: one thread per row
    {
      const T* Lkk = panel + k * kTile;
      int q = 0;   // ordinal of the owned panel tile
      for (int i = k + 1; i < nt; ++i) {
        const int t = tile_index(i, k);
        if (t % CL != rank) continue;
        if (q * TS <= tid && tid < (q + 1) * TS) {
          T* row = tiles + (t / CL) * kTile + (tid - q * TS) * TP;
          T v[TS];
#pragma unroll
          for (int c = 0; c < TS; ++c) v[c] = row[c];
#pragma unroll
          for (int c = 0; c < TS; ++c) {
            const T l = v[c] * rcs[c];
            v[c] = l;
#pragma unroll
            for (int j = c + 1; j < TS; ++j) v[j] = fma_rn<T>(-l, Lkk[j * TP + c], v[j]);
          }
#pragma unroll
          for (int c = 0; c < TS; ++c) row[c] = v[c];
        }
        ++q;
      }
    }
    __syncthreads();
    cluster.sync();
    // the panel tiles of every CTA into the local buffer (row i at panel + i * kTile)
    for (int i = k + 1; i < nt; ++i) {
      const int t = tile_index(i, k);
      const T* src = t % CL == rank ? tiles + (t / CL) * kTile
                                    : cluster.map_shared_rank(tiles + (t / CL) * kTile, t % CL);
      T* dst = panel + i * kTile;
      for (int e = tid; e < kTile; e += kThreads) dst[e] = src[e];
    }
    __syncthreads();
    // trailing tiles (i,j), k < j <= i: 4 x 4 elements a thread, 64 threads a tile
    {
      const int sub = tid >> 6;          // which of four tiles in flight
      const int w = tid & 63;
      const int r0 = (w >> 3) * 4, c0 = (w & 7) * 4;
      int q = 0;
      for (int t = rank; t < ntiles; t += CL) {
        int i = 0;
        while (tile_index(i + 1, 0) <= t) ++i;
        const int j = t - tile_index(i, 0);
        if (j <= k) continue;
        if ((q & 3) == sub) {
          T* a = tiles + (t / CL) * kTile;
          const T* li = panel + i * kTile;
          const T* lj = panel + j * kTile;
          T acc[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[u][v] = a[(r0 + u) * TP + c0 + v];
#pragma unroll 4
          for (int K = 0; K < TS; ++K) {
            T x[4], y[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              x[u] = li[(r0 + u) * TP + K];
              y[u] = lj[(c0 + u) * TP + K];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int v = 0; v < 4; ++v) acc[u][v] = fma_rn<T>(-x[u], y[v], acc[u][v]);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) a[(r0 + u) * TP + c0 + v] = acc[u][v];
        }
        ++q;
      }
    }
    __syncthreads();
  }

  // the factor back (lower triangle only) and info (the first failure over the cluster)
  for (int t = rank; t < ntiles; t += CL) {
    int i = 0;
    while (tile_index(i + 1, 0) <= t) ++i;
    const int j = t - tile_index(i, 0);
    const T* src = tiles + (t / CL) * kTile;
    for (int e = tid; e < TS * TS; e += kThreads) {
      const int r = alay == kRowMajor ? e / TS : e % TS;
      const int c = alay == kRowMajor ? e % TS : e / TS;
      const int I = i * TS + r, J = j * TS + c;
      if (I < n && J < n && I >= J) As[gidx(alay, n, I, J)] = src[r * TP + c];
    }
  }
  cluster.sync();
  if (rank == 0 && tid == 0) {
    int f = *fail;
    for (int q = 1; q < CL; ++q) {
      const int fq = *cluster.map_shared_rank(fail, q);
      f = fq < f ? fq : f;
    }
    info[s] = f == 0x7FFFFFFF ? 0 : f;
  }
  cluster.sync();   // no CTA leaves while rank 0 reads its shared memory
}

// ------------------------------------------------------------------ solve, n > 128
constexpr int RC = 8;   // right-hand sides a pass

template <typename T>
size_t big_solve_smem_bytes(int n) {
  return static_cast<size_t>(n) * RC * sizeof(T) + static_cast<size_t>(n) * TP * sizeof(T);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
potrs_big_kernel(int n, int nrhs, int layouts, int64_t batch, const T* __restrict__ L,
                 T* __restrict__ B, const int32_t* __restrict__ zinfo) {
  extern __shared__ __align__(16) unsigned char raw[];
  T* const b = reinterpret_cast<T*>(raw);     // n x RC, row-major
  T* const Ls = b + n * RC;                   // rows k*TS.. of tile column k, pitch TP
  const int64_t s = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const int alay = layouts & 1, blay = layouts >> 1;
  const int nt = (n + TS - 1) / TS;
  const T* const Lsys = L + s * static_cast<int64_t>(n) * n;
  T* const Bs = B + s * static_cast<int64_t>(n) * nrhs;
  const bool zero_x = zinfo != nullptr && __ldg(zinfo + s) != 0;

  // rows r0..n-1, columns k*TS.. of the factor into Ls (row I - r0)
  auto stage = [&](int k) {
    const int r0 = k * TS;
    const int rows = n - r0, cols = n - r0 < TS ? n - r0 : TS;
    for (int e = tid; e < rows * TS; e += kThreads) {
      const int ii = alay == kRowMajor ? e / TS : e % rows;
      const int jj = alay == kRowMajor ? e % TS : e / rows;
      if (jj < cols) Ls[ii * TP + jj] = __ldg(Lsys + gidx(alay, n, r0 + ii, r0 + jj));
    }
  };

  for (int c0 = 0; c0 < nrhs; c0 += RC) {
    const int nc = nrhs - c0 < RC ? nrhs - c0 : RC;
    for (int e = tid; e < n * RC; e += kThreads) {
      const int r = e / RC, c = e % RC;
      b[e] = c < nc ? Bs[bidx(blay, n, nrhs, r, c0 + c)] : T(0);
    }
    // forward: L y = b
    for (int k = 0; k < nt; ++k) {
      __syncthreads();
      stage(k);
      __syncthreads();
      const int r0 = k * TS;
      const int cols = n - r0 < TS ? n - r0 : TS;
      if (tid < 32) {
        T v[RC];
        const bool own = lane < cols;
#pragma unroll
        for (int c = 0; c < RC; ++c) v[c] = own ? b[(r0 + lane) * RC + c] : T(0);
        for (int K = 0; K < cols; ++K) {
          const T rk = T(1) / Ls[K * TP + K];
          if (lane == K) {
#pragma unroll
            for (int c = 0; c < RC; ++c) v[c] = v[c] * rk;
          }
          const T lrk = own ? Ls[lane * TP + K] : T(0);
#pragma unroll
          for (int c = 0; c < RC; ++c) {
            const T y = __shfl_sync(0xFFFFFFFFu, v[c], K);
            if (own && lane > K) v[c] = fma_rn<T>(-lrk, y, v[c]);
          }
        }
        if (own) {
#pragma unroll
          for (int c = 0; c < RC; ++c) b[(r0 + lane) * RC + c] = v[c];
        }
      }
      __syncthreads();
      // the rows below: 32 updates each, in increasing K
      for (int e = tid; e < (n - r0 - cols) * RC; e += kThreads) {
        const int I = r0 + cols + e / RC, c = e % RC;
        T acc = b[I * RC + c];
        const T* lrow = Ls + (I - r0) * TP;
        for (int K = 0; K < cols; ++K) acc = fma_rn<T>(-lrow[K], b[(r0 + K) * RC + c], acc);
        b[I * RC + c] = acc;
      }
    }
    // backward: L^T x = y
    for (int k = nt - 1; k >= 0; --k) {
      __syncthreads();
      stage(k);
      __syncthreads();
      const int r0 = k * TS;
      const int cols = n - r0 < TS ? n - r0 : TS;
      // the rows of this block first take the updates of the rows below, decreasing K
      for (int e = tid; e < cols * RC; e += kThreads) {
        const int J = e / RC, c = e % RC;
        T acc = b[(r0 + J) * RC + c];
        for (int K = n - 1; K >= r0 + cols; --K)
          acc = fma_rn<T>(-Ls[(K - r0) * TP + J], b[K * RC + c], acc);
        b[(r0 + J) * RC + c] = acc;
      }
      __syncthreads();
      if (tid < 32) {
        T v[RC];
        const bool own = lane < cols;
#pragma unroll
        for (int c = 0; c < RC; ++c) v[c] = own ? b[(r0 + lane) * RC + c] : T(0);
        for (int K = cols - 1; K >= 0; --K) {
          const T rk = T(1) / Ls[K * TP + K];
          if (lane == K) {
#pragma unroll
            for (int c = 0; c < RC; ++c) v[c] = v[c] * rk;
          }
          const T lkr = own ? Ls[K * TP + lane] : T(0);
#pragma unroll
          for (int c = 0; c < RC; ++c) {
            const T x = __shfl_sync(0xFFFFFFFFu, v[c], K);
            if (own && lane < K) v[c] = fma_rn<T>(-lkr, x, v[c]);
          }
        }
        if (own) {
#pragma unroll
          for (int c = 0; c < RC; ++c) b[(r0 + lane) * RC + c] = v[c];
        }
      }
    }
    __syncthreads();
    for (int e = tid; e < n * RC; e += kThreads) {
      const int r = e / RC, c = e % RC;
      if (c < nc) Bs[bidx(blay, n, nrhs, r, c0 + c)] = zero_x ? T(0) : b[e];
    }
    __syncthreads();
  }
}

}  // namespace

template <typename T>
cudaError_t launch_chol_cluster(int layout, int n, int64_t batch, T* A, int32_t* info,
                                cudaStream_t stream) {
  if (n <= 128 || n > kMaxT * TS) return cudaErrorInvalidValue;
  if (batch * CL > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const size_t bytes = cluster_smem_bytes<T>();
  cudaError_t e = cudaFuncSetAttribute(chol_cluster_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(batch * CL), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, chol_cluster_kernel<T>, n, layout & 1, batch, A, info);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_potrs_big(int layout, int n, int nrhs, int64_t batch, const T* L, T* B,
                             const int32_t* zinfo, cudaStream_t stream) {
  if (n <= 128 || n > kMaxT * TS || nrhs < 1) return cudaErrorInvalidValue;
  if (batch > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const size_t bytes = big_solve_smem_bytes<T>(n);
  cudaError_t e = cudaFuncSetAttribute(potrs_big_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  potrs_big_kernel<T><<<static_cast<unsigned>(batch), kThreads, bytes, stream>>>(
      n, nrhs, layout, batch, L, B, zinfo);
  return cudaGetLastError();
}

template cudaError_t launch_chol_cluster<float>(int, int, int64_t, float*, int32_t*,
                                                cudaStream_t);
template cudaError_t launch_chol_cluster<double>(int, int, int64_t, double*, int32_t*,
                                                 cudaStream_t);
template cudaError_t launch_potrs_big<float>(int, int, int, int64_t, const float*, float*,
                                             const int32_t*, cudaStream_t);
template cudaError_t launch_potrs_big<double>(int, int, int, int64_t, const double*, double*,
                                              const int32_t*, cudaStream_t);

}  // namespace bsolve
