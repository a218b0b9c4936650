// Cholesky for 128 < n <= 256: the lower triangle of one system spread over the shared
// memory of a thread-block cluster of four CTAs (cuSolverDx docs, "Cholesky
// Factorization", the cluster / distributed-shared-memory tiling for orders beyond one
// CTA), and the solve with the stored factor, one CTA per system.
//
// Factor: the lower triangle in 32 x 32 tiles; tile t = i(i+1)/2 + j of tile row i and
// tile column j <= i lives in CTA t % 4, slot t / 4. Right-looking by tile columns k. The
// FP64 pipe charges a warp instruction whatever its active lanes and each SM sub-partition
// has its own, so the serial work of a step (the diagonal tile, the panel, the next tile
// column) runs on teams of four warps, one per sub-partition, that split each tile's
// columns (or rows) between them:
//   1. the owner of tile (k,k) factors it with a team (lane r holds row r of the tile in
//      shared memory, warp u the columns j = u mod 4; column c: its warp takes
//      l_cc = sqrt(a_cc), r_c = 1/l_cc and scales the column, the team synchronizes, then
//      each warp applies the column to its own columns, a_rj -= l_rc l_jc for c < j <= r;
//      the warp of column c+1 applies column c to it first and takes its square root at
//      once, so the chain overlaps the team's remaining updates);
//   2. cluster barrier; every CTA copies L_kk and the reciprocals out of the owner's
//      shared memory (distributed shared memory loads) and solves its own panel tiles
//      (i,k), i > k, one team a tile, in the same column-split order (l_rc = a_rc r_c,
//      then a_rj -= l_rc l_jc for the tile's later columns);
//   3. cluster barrier; the tiles (i,k+1) of the next tile column take the panel's 32
//      updates first, one team a tile (each warp eight rows), then (look-ahead) a team of
//      the owner of tile (k+1,k+1) factors it while every other warp applies the panel to
//      the remaining trailing tiles (i,j), k+1 < j <= i, one warp a tile, taken from a
//      shared counter (the factoring team joins when it is done). Element (r, c) takes
//      a_rc -= l_rK l_cK in increasing K. FP64 reads the panel tiles where they live (the
//      other CTAs' through distributed-shared-memory loads: an FP64 update costs the pipe
//      far more than its loads, and no staging buffer keeps two CTAs per SM); FP32 stages
//      them.
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
constexpr int kWarps = kThreads / 32;
constexpr int kTeam = 4;                 // warps of a team: one per SM sub-partition
constexpr int kTeams = kWarps / kTeam;
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

// FP32 stages the panel tile column in local shared memory (its updates are cheap, remote
// loads would dominate); FP64 reads the panel tiles where they live (each FP64 update
// costs the pipe far more than its loads, and no staging keeps two CTAs per SM).
template <typename T>
constexpr bool kStagePanel = sizeof(T) == 4;

template <typename T>
size_t cluster_smem_bytes() {
  // owned tiles, a staged copy of L_kk, the staged panel (FP32), the diagonal
  // reciprocals (own and staged), the first failure and the trailing-tile counter
  return static_cast<size_t>(kMaxSlots + 1 + (kStagePanel<T> ? kMaxT : 0)) * kTile * sizeof(T) +
         2 * TS * sizeof(T) + 16;
}

// One warp applies the 32 updates of a panel to a 32 x 32 tile: a_rc -= l_iK l_jK for
// K = 0..31 in order, li / lj the panel tiles of the tile's row and column (pitch TP);
// lane = a 4 x 4 block of each half of the tile (rows 0-15, then 16-31).
template <typename T>
__device__ __forceinline__ void update_tile(T* a, const T* li, const T* lj, int lane) {
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    const int r0 = h * 16 + (lane >> 3) * 4, c0 = (lane & 7) * 4;
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
}

__device__ __forceinline__ void tile_coords(int t, int& i, int& j) {
  i = 0;
  while (tile_index(i + 1, 0) <= t) ++i;
  j = t - tile_index(i, 0);
}

// Barrier of the four warps of team `team` (named barriers 1 and 2, immediate ids; 0 is
// __syncthreads).
static_assert(kTeams == 2, "one named barrier per team");
__device__ __forceinline__ void team_sync(int team) {
  if (team == 0)
    asm volatile("bar.sync 1, %0;" ::"n"(kTeam * 32) : "memory");
  else
    asm volatile("bar.sync 2, %0;" ::"n"(kTeam * 32) : "memory");
}

// The first column j > c that warp u of a team owns (j = u mod 4).
__device__ __forceinline__ int first_col(int c, int u) { return c + 1 + ((u - c - 1) & (kTeam - 1)); }

// Factor the diagonal tile at `a` (pitch TP, in shared memory) with a team of four warps
// (this thread's warp is u of team `team`); lane r owns row r, warp u the columns j = u
// mod 4. k is the tile column (for the global index of a failing minor), n the order.
// Every element (r, j), j <= r, takes a_rj -= l_rc l_jc for c = 0, 1, ... in order, one
// fused multiply-add each, and the diagonal and column steps of the CPU oracle.
template <typename T>
__device__ void potrf_tile_team(T* a, T* rc, int k, int n, int* fail, int team, int u) {
  const int r = threadIdx.x & 31;
  int first = 0x7FFFFFFF;
  // column c's pivot and scaling, by the warp that owns column c
  auto pivot = [&](int c) {
    const T d = a[c * TP + c];
    if (!(d > T(0)) && k * TS + c < n && first == 0x7FFFFFFF) first = k * TS + c + 1;
    const T l = sqrt_rn<T>(d);
    const T rr = rcp_rn<T>(l);
    __syncwarp();   // every lane has read a_cc
    if (r == c) a[c * TP + c] = l;
    if (r > c) a[r * TP + c] = a[r * TP + c] * rr;
    if (r == 0) rc[c] = rr;
  };
  if (u == 0) pivot(0);
  team_sync(team);
#pragma unroll 1
  for (int c = 0; c < TS; ++c) {
    const T lrc = a[r * TP + c];
    const int cn = c + 1;
    // look-ahead: the warp of column c+1 applies column c to it and takes its pivot first
    if (cn < TS && (cn & (kTeam - 1)) == u) {
      if (r >= cn) a[r * TP + cn] = fma_rn<T>(-lrc, a[cn * TP + c], a[r * TP + cn]);
      __syncwarp();
      pivot(cn);
    }
#pragma unroll 1
    for (int j = first_col(c, u); j < TS; j += kTeam) {
      if (j == cn) continue;
      if (r >= j) a[r * TP + j] = fma_rn<T>(-lrc, a[j * TP + c], a[r * TP + j]);
    }
    team_sync(team);   // column c+1 is scaled; column c applied everywhere
  }
  if (r == 0 && first != 0x7FFFFFFF) atomicMin(fail, first);
}

// Solve a panel tile in place with a team: row r of the tile (lane r) becomes
// L_rk = A_rk L_kk^-T, column by column (l_rc = a_rc r_c, then a_rj -= l_rc (L_kk)_jc for
// the later columns j of warp u's residue), the oracle's order for every element. `lkk` is
// the factored diagonal tile (pitch TP), `rcs` its diagonal reciprocals.
template <typename T>
__device__ void panel_tile_team(T* a, const T* lkk, const T* rcs, int team, int u) {
  const int r = threadIdx.x & 31;
  T* const row = a + r * TP;
  if (u == 0) row[0] = row[0] * rcs[0];
  team_sync(team);
#pragma unroll 1
  for (int c = 0; c < TS; ++c) {
    const T lrc = row[c];
    const int cn = c + 1;
    if (cn < TS && (cn & (kTeam - 1)) == u) {
      row[cn] = fma_rn<T>(-lrc, lkk[cn * TP + c], row[cn]);
      row[cn] = row[cn] * rcs[cn];
    }
#pragma unroll 1
    for (int j = first_col(c, u); j < TS; j += kTeam) {
      if (j == cn) continue;
      row[j] = fma_rn<T>(-lrc, lkk[j * TP + c], row[j]);
    }
    team_sync(team);
  }
}

// One warp of a team applies the 32 updates of a panel to rows 8u..8u+7 of a 32 x 32 tile
// (a_rc -= l_iK l_jK for K = 0..31 in order); lane = a 2 x 4 block.
template <typename T>
__device__ __forceinline__ void update_rows_team(T* a, const T* li, const T* lj, int lane, int u) {
  const int r0 = 8 * u + (lane >> 3) * 2, c0 = (lane & 7) * 4;
  T acc[2][4];
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int v = 0; v < 4; ++v) acc[p][v] = a[(r0 + p) * TP + c0 + v];
#pragma unroll 4
  for (int K = 0; K < TS; ++K) {
    T x[2], y[4];
#pragma unroll
    for (int p = 0; p < 2; ++p) x[p] = li[(r0 + p) * TP + K];
#pragma unroll
    for (int v = 0; v < 4; ++v) y[v] = lj[(c0 + v) * TP + K];
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[p][v] = fma_rn<T>(-x[p], y[v], acc[p][v]);
  }
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int v = 0; v < 4; ++v) a[(r0 + p) * TP + c0 + v] = acc[p][v];
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
chol_cluster_kernel(int n, int alay, int64_t batch, T* __restrict__ A, int32_t* __restrict__ info) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int64_t s = blockIdx.x / CL;
  extern __shared__ __align__(16) unsigned char raw[];
  T* const tiles = reinterpret_cast<T*>(raw);
  T* const lkk = tiles + kMaxSlots * kTile;  // staged L_kk
  T* const panel = lkk + kTile;              // FP32: the staged panel tiles (i,k) at row i
  T* const rc = panel + (kStagePanel<T> ? kMaxT : 0) * kTile;   // reciprocals of the tile
                                                                // this CTA factored
  T* const rcs = rc + TS;                  // staged reciprocals of L_kk
  int* const fail = reinterpret_cast<int*>(rcs + TS);
  int* const next = fail + 1;              // the trailing-tile counter of a step
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

  const int warp = tid >> 5, lane = tid & 31;
  // the panel tile (i,k): local, staged (FP32) or remote (FP64)
  auto panel_tile = [&](int i, int k) -> const T* {
    if constexpr (kStagePanel<T>) {
      return panel + i * kTile;
    } else {
      const int t = tile_index(i, k);
      return cluster.map_shared_rank(tiles + (t / CL) * kTile, t % CL);
    }
  };
  const int team = warp / kTeam, u = warp % kTeam;   // warp u of a team runs on sub-partition u
  // tile (0,0) lives in rank 0, slot 0
  if (rank == 0 && team == 0) potrf_tile_team<T>(tiles, rc, 0, n, fail, team, u);
  for (int k = 0; k < nt; ++k) {
    const int tkk = tile_index(k, k);
    cluster.sync();   // L_kk is factored
    // L_kk and its reciprocals from the owner
    {
      const T* src = cluster.map_shared_rank(tiles + (tkk / CL) * kTile, tkk % CL);
      for (int e = tid; e < kTile; e += kThreads) lkk[e] = src[e];
      const T* rsrc = cluster.map_shared_rank(rc, tkk % CL);
      if (tid < TS) rcs[tid] = rsrc[tid];
    }
    __syncthreads();
    // the owned panel tiles (i,k), i > k: one team a tile
    {
      int q = 0;   // ordinal of the owned panel tile
      for (int i = k + 1; i < nt; ++i) {
        const int t = tile_index(i, k);
        if (t % CL != rank) continue;
        if (q % kTeams == team) panel_tile_team<T>(tiles + (t / CL) * kTile, lkk, rcs, team, u);
        ++q;
      }
    }
    __syncthreads();
    cluster.sync();   // the panel tiles (i,k) are final
    if constexpr (kStagePanel<T>) {
      for (int i = k + 1; i < nt; ++i) {
        const int t = tile_index(i, k);
        const T* src = cluster.map_shared_rank(tiles + (t / CL) * kTile, t % CL);
        for (int e = tid; e < kTile; e += kThreads) panel[i * kTile + e] = src[e];
      }
      __syncthreads();
    }
    // look-ahead: the next tile column first (one team a tile, eight rows a warp) ...
    if (k + 1 < nt) {
      int q = 0;
      for (int i = k + 1; i < nt; ++i) {
        const int t = tile_index(i, k + 1);
        if (t % CL != rank) continue;
        if (q % kTeams == team)
          update_rows_team<T>(tiles + (t / CL) * kTile, panel_tile(i, k), panel_tile(k + 1, k),
                              lane, u);
        ++q;
      }
    }
    if (tid == 0) *next = 0;
    __syncthreads();
    // ... then a team of the next diagonal tile's owner factors it while the other warps
    // apply this panel to the remaining trailing tiles, one warp a tile from the counter
    // (the team takes tiles too once it is done)
    const int tn = tile_index(k + 1, k + 1);
    if (k + 1 < nt && tn % CL == rank && team == 0)
      potrf_tile_team<T>(tiles + (tn / CL) * kTile, rc, k + 1, n, fail, team, u);
    {
      // the owned trailing tiles, in slot order: t = rank + CL * slot with column j > k + 1
#pragma unroll 1
      for (;;) {
        int idx = 0;
        if (lane == 0) idx = atomicAdd(next, 1);
        idx = __shfl_sync(0xFFFFFFFFu, idx, 0);
        int t = rank, i = 0, j = 0, seen = -1;
        for (; t < ntiles; t += CL) {
          tile_coords(t, i, j);
          if (j > k + 1 && ++seen == idx) break;
        }
        if (t >= ntiles) break;
        update_tile<T>(tiles + (t / CL) * kTile, panel_tile(i, k), panel_tile(j, k), lane);
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
template <typename T>
size_t big_solve_smem_bytes(int n, int rc) {
  return static_cast<size_t>(n) * rc * sizeof(T) + static_cast<size_t>(n) * TP * sizeof(T);
}

// RC right-hand sides a pass (1, 2, 4 or 8: the call's count, up to 8), row-major in
// shared memory; the diagonal reciprocals of a tile taken by its 32 lanes at once.
template <typename T, int RC>
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
        // y_K = b_K * (1/l_KK): the 32 reciprocals at once, one per lane
        const T rmine = own ? T(1) / Ls[lane * TP + lane] : T(1);
#pragma unroll
        for (int c = 0; c < RC; ++c) v[c] = own ? b[(r0 + lane) * RC + c] : T(0);
        for (int K = 0; K < cols; ++K) {
          const T rk = __shfl_sync(0xFFFFFFFFu, rmine, K);
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
      // the rows below: 32 updates each, in increasing K (only the call's columns)
      for (int e = tid; e < (n - r0 - cols) * nc; e += kThreads) {
        const int I = r0 + cols + e / nc, c = e % nc;
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
      for (int e = tid; e < cols * nc; e += kThreads) {
        const int J = e / nc, c = e % nc;
        T acc = b[(r0 + J) * RC + c];
        for (int K = n - 1; K >= r0 + cols; --K)
          acc = fma_rn<T>(-Ls[(K - r0) * TP + J], b[K * RC + c], acc);
        b[(r0 + J) * RC + c] = acc;
      }
      __syncthreads();
      if (tid < 32) {
        T v[RC];
        const bool own = lane < cols;
        const T rmine = own ? T(1) / Ls[lane * TP + lane] : T(1);
#pragma unroll
        for (int c = 0; c < RC; ++c) v[c] = own ? b[(r0 + lane) * RC + c] : T(0);
        for (int K = cols - 1; K >= 0; --K) {
          const T rk = __shfl_sync(0xFFFFFFFFu, rmine, K);
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

template <typename T, int RC>
cudaError_t launch_big_rc(int layout, int n, int nrhs, int64_t batch, const T* L, T* B,
                          const int32_t* zinfo, cudaStream_t stream) {
  const size_t bytes = big_solve_smem_bytes<T>(n, RC);
  cudaError_t e = cudaFuncSetAttribute(potrs_big_kernel<T, RC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  potrs_big_kernel<T, RC><<<static_cast<unsigned>(batch), kThreads, bytes, stream>>>(
      n, nrhs, layout, batch, L, B, zinfo);
  return cudaGetLastError();
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
  if (nrhs == 1) return launch_big_rc<T, 1>(layout, n, nrhs, batch, L, B, zinfo, stream);
  if (nrhs == 2) return launch_big_rc<T, 2>(layout, n, nrhs, batch, L, B, zinfo, stream);
  if (nrhs <= 4) return launch_big_rc<T, 4>(layout, n, nrhs, batch, L, B, zinfo, stream);
  return launch_big_rc<T, 8>(layout, n, nrhs, batch, L, B, zinfo, stream);
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
