// Solves with a stored factor: getrs (L\U from getrf and its swap sequence) and potrs
// (the lower Cholesky factor from potrf). "Factor once, call this per right-hand side"
// (GLASS API reference, "Block-tridiagonal Ops", bdsv_solve; TDLS API,
// "solver_static.hpp File Reference", separate substitution).
//
// n <= 32: one system per group of G = NT / R lanes (32/G systems per warp), lane t owns
// positions p = t + qG (q < R): their right-hand-side rows in registers, and in registers
// the factor entries those rows need. For LU that is row p of L\U (the forward sweep
// reads l_pk, k < p, the backward sweep u_pk, k > p). For Cholesky the forward sweep
// needs row p of L and the backward sweep (with L^T) column p, so the lane holds the
// symmetric fill of the lower triangle: v[j] = L[max(p,j)][min(p,j)] (row p left of the
// diagonal, column p right of it). Each step k broadcasts one value per right-hand side
// from the owner of position k by a shuffle, and every lane applies it from registers:
// no shared memory, no barrier.
// 32 < n <= 128: one warp per system, the factor in shared memory with an odd pitch, lane
// t owning positions t, t+32, ...
//
// getrs: lane t loads the right-hand-side row that the swap sequence brings to position
// t (the swaps undone from the last: pos = t, then for k = n-1..0 pos <- tau_k(pos)); an
// ipiv entry outside 1..n swaps nothing, so no access leaves the system.
// The mirror solve (the row-major reading of TDLS, factor of S = A^T): the lane of
// position p holds column p of S, a contiguous row of the stored array; U^T z = b runs
// like the Cholesky forward sweep (z_k = b_k r_k at the owner, then b_j -= s_kj z_k for
// j > k), L^T w = z like the LU backward sweep without the scaling, and x = P^T w is the
// store: the value of position p goes to the row the swaps bring to p.
// The arithmetic is the CPU oracle's, operation by operation: b_i -= l_ik y_k for i > k
// in increasing k (Cholesky: y_k = b_k * (1/l_kk) first), then x_k = y_k * r_k and
// b_i -= m_ik x_k for i < k in decreasing k; r_k = 1/u_kk (1 for a pivot below the
// smallest normal) for LU, 1/l_kk for Cholesky; every update one fused multiply-add.
#include <cfloat>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace bsolve {
namespace {

// kSolveLuT: the mirror solve of the row-major reading of an LU factor (TDLS API,
// "solver_static.hpp File Reference": the factor is of S, the stored array read
// column-major, P S = L U with S = A^T; then U^T z = b, L^T w = z, x = P^T w).
enum SolveKind : int { kSolveLu = 0, kSolveChol = 1, kSolveLuT = 2 };

// Positions per lane for the order tiers 8, 16 and 32. Two positions per lane halve the
// shuffles per system and let a step skip, at compile time, a slot whose rows are all
// past (FP32 n=16 getrs: 35.5 -> 31.4 us; FP64 n=32 potrs: 1.97 -> 1.33 ms; four per lane
// gained nothing more).
constexpr int kRows8 = 2, kRows16 = 2, kRows32 = 2;

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;

template <typename T> struct Floor;   // smallest normal number: a smaller |pivot| is singular
template <> struct Floor<float> {
  __device__ __forceinline__ static float v() { return FLT_MIN; }
};
template <> struct Floor<double> {
  __device__ __forceinline__ static double v() { return DBL_MIN; }
};

template <typename T, int KIND>
__device__ __forceinline__ T diag_rcp(T d) {
  if (KIND != kSolveChol) return (fabs(d) >= Floor<T>::v()) ? T(1) / d : T(1);
  return T(1) / d;
}

// Element (r, c) of an n x m matrix in the given storage order.
__device__ __forceinline__ int64_t idx(int layout, int rows, int cols, int r, int c) {
  return layout == kRowMajor ? static_cast<int64_t>(r) * cols + c
                             : static_cast<int64_t>(c) * rows + r;
}

// ------------------------------------------------------------------ n <= 32, registers
// R positions per lane: lane t of a group of G = NT / R lanes owns positions t + q G.
template <typename T, int N>
__device__ __forceinline__ void ldg_row(const T* __restrict__ p, T (&r)[N]) {
  if constexpr ((N * sizeof(T)) % 16 == 0) {
#pragma unroll
    for (int j = 0; j < N; j += 16 / sizeof(T)) {
      if constexpr (std::is_integral<T>::value) {
        const int4 v = __ldg(reinterpret_cast<const int4*>(p + j));
        r[j] = v.x; r[j + 1] = v.y; r[j + 2] = v.z; r[j + 3] = v.w;
      } else if constexpr (sizeof(T) == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p + j));
        r[j] = v.x; r[j + 1] = v.y; r[j + 2] = v.z; r[j + 3] = v.w;
      } else {
        const double2 v = __ldg(reinterpret_cast<const double2*>(p + j));
        r[j] = v.x; r[j + 1] = v.y;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) r[j] = __ldg(p + j);
  }
}

// A row of N elements in 32-byte pieces (sm_100 and later; p 32-byte aligned, the factor
// read only).
template <typename T, int N>
__device__ __forceinline__ void ldg_row32(const T* __restrict__ p, T (&r)[N]) {
  static_assert((N * sizeof(T)) % 32 == 0, "whole 32-byte pieces");
#pragma unroll
  for (int j = 0; j < N; j += 32 / sizeof(T)) {
    if constexpr (sizeof(T) == 4) {
      asm("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
          : "=f"(r[j]), "=f"(r[j + 1]), "=f"(r[j + 2]), "=f"(r[j + 3]), "=f"(r[j + 4]),
            "=f"(r[j + 5]), "=f"(r[j + 6]), "=f"(r[j + 7])
          : "l"(p + j));
    } else {
      asm("ld.global.nc.v4.f64 {%0,%1,%2,%3}, [%4];"
          : "=d"(r[j]), "=d"(r[j + 1]), "=d"(r[j + 2]), "=d"(r[j + 3])
          : "l"(p + j));
    }
  }
}

// layouts: bit 0 the factor's storage order, bit 1 B's, bit 2 (FULL instances) the factor
// 32-byte aligned, its rows then read in 32-byte pieces
template <typename T, int NT, int R, int RT, int KIND, bool FULL>
__global__ void __launch_bounds__(kThreads)
solve_reg_kernel(int n_, int nrhs_, int layouts_, int64_t batch, const T* __restrict__ M,
                 const int32_t* __restrict__ ipiv, T* __restrict__ B,
                 const int32_t* __restrict__ zinfo) {
  constexpr int G = NT / R;
  constexpr int GPW = 32 / G;
  const int n = FULL ? NT : n_;
  const int nrhs = FULL ? RT : nrhs_;
  const int layouts = layouts_ & 3;
  const bool w32 = FULL && (layouts_ & 4) != 0;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane / G;
  const int t = lane % G;
  const int64_t s = (static_cast<int64_t>(blockIdx.x) * kWarps + warp) * GPW + g;
  const bool valid = s < batch;
  const T* Ms = M + s * n * n;
  T* Bs = B + s * n * nrhs;

  bool ok[R];
  int src[R];   // the right-hand-side row that lands at position t + qG
#pragma unroll
  for (int q = 0; q < R; ++q) {
    ok[q] = valid && (FULL || t + q * G < n);
    src[q] = t + q * G;
  }
  // LU with row-major B in one pass: every lane loads its own rows of B (rows t + qG) with
  // the factor and the swap sequence, and takes the permuted rows from the group's lanes by
  // shuffles once the swaps are known, instead of a second round trip to memory that would
  // wait on the swap sequence
  constexpr bool kEarlyB = KIND == kSolveLu && FULL;
  const bool early_b = kEarlyB && (layouts >> 1) == kRowMajor;
  T bown[R][RT];
  if (kEarlyB && early_b) {
#pragma unroll
    for (int q = 0; q < R; ++q) {
      if (ok[q]) ldg_row<T, RT>(Bs + static_cast<int64_t>(t + q * G) * RT, bown[q]);
      else {
#pragma unroll
        for (int c = 0; c < RT; ++c) bown[q][c] = T(0);
      }
    }
  }
  if (KIND != kSolveChol && valid) {
    // the swaps undone from the last, on the group's copy of the swap sequence
    int iv[NT];
    if (FULL && (NT % 4) == 0) {
      ldg_row<int, NT>(ipiv + s * n, iv);
    } else {
#pragma unroll
      for (int k = 0; k < NT; ++k) iv[k] = k < n ? __ldg(ipiv + s * n + k) : k + 1;
    }
#pragma unroll
    for (int k = NT - 1; k >= 0; --k) {
      int p = iv[k] - 1;
      if (p < 0 || p >= n) p = k;   // an entry out of range swaps nothing
#pragma unroll
      for (int q = 0; q < R; ++q) {
        if (src[q] == k) src[q] = p;
        else if (src[q] == p) src[q] = k;
      }
    }
  }
  T v[R][NT];
  T rt[R];
#pragma unroll
  for (int q = 0; q < R; ++q) {
    const int pq = t + q * G;
    rt[q] = T(1);
    if (ok[q]) {
      if (FULL && ((KIND == kSolveLu && (layouts & 1) == kRowMajor) ||
                   (KIND == kSolveLuT && (layouts & 1) == kColMajor))) {
        if constexpr ((NT * sizeof(T)) % 32 == 0) {
          if (w32) ldg_row32<T, NT>(Ms + static_cast<int64_t>(pq) * NT, v[q]);
          else ldg_row<T, NT>(Ms + static_cast<int64_t>(pq) * NT, v[q]);
        } else {
          ldg_row<T, NT>(Ms + static_cast<int64_t>(pq) * NT, v[q]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          if (FULL || j < n) {
            // LU: row pq; LuT: column pq of S; Cholesky: the symmetric fill of L
            const bool rowp = KIND == kSolveLu || (KIND == kSolveChol && j <= pq);
            const int r = rowp ? pq : j;
            const int c = rowp ? j : pq;
            v[q][j] = __ldg(Ms + idx(layouts & 1, n, n, r, c));
          } else {
            v[q][j] = T(0);
          }
        }
      }
      rt[q] = diag_rcp<T, KIND>(__ldg(Ms + idx(layouts & 1, n, n, pq, pq)));
    } else {
#pragma unroll
      for (int j = 0; j < NT; ++j) v[q][j] = T(0);
    }
  }
  // a failed factor of the fused call with more right-hand sides than a tier: X = 0
  const bool zero_x = zinfo != nullptr && valid && __ldg(zinfo + s) != 0;

  // the right-hand sides RT columns at a time (one pass when nrhs <= RT)
  for (int c0 = 0; c0 < nrhs; c0 += RT) {
  T b[R][RT];
#pragma unroll
  for (int q = 0; q < R; ++q) {
    if (kEarlyB && early_b) {
      // row src[q] sits in lane src[q] % G of the group, slot src[q] / G (every lane of the
      // group joins the shuffles; rows past a partial last system are zeros, never used)
      const int sl = src[q] % G, sq = src[q] / G;
#pragma unroll
      for (int c = 0; c < RT; ++c) {
        T got = T(0);
#pragma unroll
        for (int u = 0; u < R; ++u) {
          const T v_u = __shfl_sync(0xFFFFFFFFu, bown[u][c], sl, G);
          got = sq == u ? v_u : got;
        }
        b[q][c] = ok[q] ? got : T(0);
      }
      continue;
    }
    if (ok[q]) {
      // LU: the row the swaps bring to position pq; LuT: row pq (swapped on the way out)
      const int lrow = KIND == kSolveLuT ? t + q * G : src[q];
      if (FULL && (layouts >> 1) == kRowMajor) {
        ldg_row<T, RT>(Bs + static_cast<int64_t>(lrow) * RT, b[q]);
      } else {
#pragma unroll
        for (int c = 0; c < RT; ++c)
          b[q][c] = (c0 + c < nrhs) ? Bs[idx(layouts >> 1, n, nrhs, lrow, c0 + c)] : T(0);
      }
    } else {
#pragma unroll
      for (int c = 0; c < RT; ++c) b[q][c] = T(0);
    }
  }

  // forward: L y = P b (unit L), L y = b or U^T z = b. Slot q holds positions qG..qG+G-1: it has
  // rows below k unless qG + G - 1 <= k (known at compile time).
#pragma unroll
  for (int k = 0; k < NT; ++k) {
    if (!FULL && k >= n) break;
    const int kq = k / G, kl = k % G;
    if (KIND != kSolveLu && t == kl) {
#pragma unroll
      for (int c = 0; c < RT; ++c) b[kq][c] = b[kq][c] * rt[kq];
    }
    T y[RT];
#pragma unroll
    for (int c = 0; c < RT; ++c) y[c] = __shfl_sync(0xFFFFFFFFu, b[kq][c], kl, G);
#pragma unroll
    for (int q = 0; q < R; ++q) {
      if (q * G + G - 1 <= k) continue;
      if (ok[q] && t + q * G > k) {
#pragma unroll
        for (int c = 0; c < RT; ++c) b[q][c] = fma_rn<T>(-v[q][k], y[c], b[q][c]);
      }
    }
  }
  // backward: U x = y, L^T x = y or L^T w = z (unit L). Slot q has rows above k unless
  // qG >= k.
#pragma unroll
  for (int k = NT - 1; k >= 0; --k) {
    if (!FULL && k >= n) continue;
    const int kq = k / G, kl = k % G;
    if (KIND != kSolveLuT && t == kl) {
#pragma unroll
      for (int c = 0; c < RT; ++c) b[kq][c] = b[kq][c] * rt[kq];
    }
    T x[RT];
#pragma unroll
    for (int c = 0; c < RT; ++c) x[c] = __shfl_sync(0xFFFFFFFFu, b[kq][c], kl, G);
#pragma unroll
    for (int q = 0; q < R; ++q) {
      if (q * G >= k) continue;
      if (ok[q] && t + q * G < k) {
#pragma unroll
        for (int c = 0; c < RT; ++c) b[q][c] = fma_rn<T>(-v[q][k], x[c], b[q][c]);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < R; ++q) {
    if (!ok[q]) continue;
    const int pq = KIND == kSolveLuT ? src[q] : t + q * G;   // LuT: x = P^T w
    if (FULL && (layouts >> 1) == kRowMajor && (RT * sizeof(T)) % 16 == 0) {
      T* dst = Bs + static_cast<int64_t>(pq) * RT;
#pragma unroll
      for (int c = 0; c < RT; c += 16 / sizeof(T)) {
        if constexpr (sizeof(T) == 4)
          *reinterpret_cast<float4*>(dst + c) =
              zero_x ? make_float4(0.f, 0.f, 0.f, 0.f)
                     : make_float4(b[q][c], b[q][c + 1], b[q][c + 2], b[q][c + 3]);
        else
          *reinterpret_cast<double2*>(dst + c) =
              zero_x ? make_double2(0.0, 0.0) : make_double2(b[q][c], b[q][c + 1]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < RT; ++c)
        if (c0 + c < nrhs) Bs[idx(layouts >> 1, n, nrhs, pq, c0 + c)] = zero_x ? T(0) : b[q][c];
    }
  }
  }   // right-hand-side chunk
}

template <typename T, int NT, int R, int RT, int KIND>
cudaError_t launch_reg_tier(int layout, int n, int nrhs, int64_t batch, const T* M,
                            const int32_t* ipiv, T* B, const int32_t* zinfo,
                            cudaStream_t stream) {
  constexpr int per_block = kWarps * (32 / (NT / R));
  const int64_t blocks = (batch + per_block - 1) / per_block;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const unsigned nb = static_cast<unsigned>(blocks);
  if (n == NT && nrhs == RT)
    solve_reg_kernel<T, NT, R, RT, KIND, true><<<nb, kThreads, 0, stream>>>(
        n, nrhs, layout | (reinterpret_cast<uintptr_t>(M) % 32 == 0 ? 4 : 0), batch, M, ipiv, B,
        zinfo);
  else
    solve_reg_kernel<T, NT, R, RT, KIND, false><<<nb, kThreads, 0, stream>>>(n, nrhs, layout, batch, M, ipiv, B, zinfo);
  return cudaGetLastError();
}

template <typename T, int NT, int R, int KIND>
cudaError_t launch_reg_rhs(int layout, int n, int nrhs, int64_t batch, const T* M,
                           const int32_t* ipiv, T* B, const int32_t* zinfo, cudaStream_t stream) {
  if (nrhs <= 1) return launch_reg_tier<T, NT, R, 1, KIND>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream);
  if (nrhs <= 2) return launch_reg_tier<T, NT, R, 2, KIND>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream);
  if (nrhs <= 4) return launch_reg_tier<T, NT, R, 4, KIND>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream);
  return launch_reg_tier<T, NT, R, 8, KIND>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream);
}

// ---------------------------------------- 32 < n <= 128, shared memory, one warp a system
__host__ __device__ inline int odd_pitch(int n) { return n | 1; }

// Q positions per lane (lane t owns t, t+32, ...): Q = 2 for n <= 64, 4 for n <= 128.
template <typename T, int Q>
__device__ __forceinline__ T pick(const T (&v)[Q], int q) {
  T r = v[0];
#pragma unroll
  for (int i = 1; i < Q; ++i) r = (q == i) ? v[i] : r;
  return r;
}

// ilv: the element stride of TDLS's interleaved batched layouts (element e of system s at
// base_s[e * ilv], base_s = (s / ilv) * ilv * size + s % ilv, for the factor, B and
// ipiv); 1 for the plain layout, where the offsets are the plain ones.
template <typename T, int RT, int KIND, int Q, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
solve_smem_kernel(int n, int nrhs, int layouts, int64_t batch, const T* __restrict__ M,
                  const int32_t* __restrict__ ipiv, T* __restrict__ B,
                  const int32_t* __restrict__ zinfo, int64_t ilv) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int P = odd_pitch(n);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t s = static_cast<int64_t>(blockIdx.x) * WARPS + warp;
  if (s >= batch) return;   // whole warp: no block barrier below
  T* const F = reinterpret_cast<T*>(smem_raw) + static_cast<int64_t>(warp) * n * P;
  const int64_t blk = s / ilv, sl = s - blk * ilv;
  const T* Ms = M + blk * ilv * n * n + sl;
  T* Bs = B + blk * ilv * n * nrhs + sl;
  const int32_t* ips = ipiv == nullptr ? nullptr : ipiv + blk * ilv * n + sl;

  // the factor (LU: all of it; Cholesky: the lower triangle only)
  for (int e = lane; e < n * n; e += 32) {
    int r, c;
    if ((layouts & 1) == kRowMajor) {
      r = e / n;
      c = e - r * n;
    } else {
      c = e / n;
      r = e - c * n;
    }
    if (KIND != kSolveChol || c <= r) cp_async_elem<T>(F + r * P + c, Ms + e * ilv);
  }
  cp_async_wait_all();
  __syncwarp();

  int src[Q];
#pragma unroll
  for (int q = 0; q < Q; ++q) src[q] = lane + 32 * q;
  if (KIND != kSolveChol) {
    int ip[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q)
      ip[q] = lane + 32 * q < n ? __ldg(ips + static_cast<int64_t>(lane + 32 * q) * ilv) - 1 : 0;
    for (int k = n - 1; k >= 0; --k) {
      int p = __shfl_sync(0xFFFFFFFFu, pick<int, Q>(ip, k >> 5), k & 31);
      if (p < 0 || p >= n) p = k;   // an entry out of range swaps nothing
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        if (src[q] == k) src[q] = p;
        else if (src[q] == p) src[q] = k;
      }
    }
  }
  T rq[Q];
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int i = lane + 32 * q;
    rq[q] = i < n ? diag_rcp<T, KIND>(F[i * P + i]) : T(1);
  }
  const bool zero_x = zinfo != nullptr && __ldg(zinfo + s) != 0;

  // the right-hand sides RT columns at a time
  for (int c0 = 0; c0 < nrhs; c0 += RT) {
    T b[Q][RT];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const bool ok = lane + 32 * q < n;
      const int lrow = KIND == kSolveLuT ? lane + 32 * q : src[q];
#pragma unroll
      for (int c = 0; c < RT; ++c)
        b[q][c] = (ok && c0 + c < nrhs) ? Bs[idx(layouts >> 1, n, nrhs, lrow, c0 + c) * ilv]
                                        : T(0);
    }
    for (int k = 0; k < n; ++k) {
      const int kq = k >> 5, kl = k & 31;
      if (KIND != kSolveLu && lane == kl) {
#pragma unroll
        for (int q = 0; q < Q; ++q)
          if (q == kq)
#pragma unroll
            for (int c = 0; c < RT; ++c) b[q][c] = b[q][c] * rq[q];
      }
      T y[RT];
#pragma unroll
      for (int c = 0; c < RT; ++c) {
        T own = b[0][c];
#pragma unroll
        for (int q = 1; q < Q; ++q) own = (kq == q) ? b[q][c] : own;
        y[c] = __shfl_sync(0xFFFFFFFFu, own, kl);
      }
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const int i = lane + 32 * q;
        if (i > k && i < n) {
          const T l = KIND == kSolveLuT ? F[k * P + i] : F[i * P + k];
#pragma unroll
          for (int c = 0; c < RT; ++c) b[q][c] = fma_rn<T>(-l, y[c], b[q][c]);
        }
      }
    }
    for (int k = n - 1; k >= 0; --k) {
      const int kq = k >> 5, kl = k & 31;
      if (KIND != kSolveLuT && lane == kl) {
#pragma unroll
        for (int q = 0; q < Q; ++q)
          if (q == kq)
#pragma unroll
            for (int c = 0; c < RT; ++c) b[q][c] = b[q][c] * rq[q];
      }
      T x[RT];
#pragma unroll
      for (int c = 0; c < RT; ++c) {
        T own = b[0][c];
#pragma unroll
        for (int q = 1; q < Q; ++q) own = (kq == q) ? b[q][c] : own;
        x[c] = __shfl_sync(0xFFFFFFFFu, own, kl);
      }
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const int i = lane + 32 * q;
        if (i < k) {
          const T u = KIND == kSolveLu ? F[i * P + k] : F[k * P + i];
#pragma unroll
          for (int c = 0; c < RT; ++c) b[q][c] = fma_rn<T>(-u, x[c], b[q][c]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const int i = lane + 32 * q;
      if (i < n) {
        const int srow = KIND == kSolveLuT ? src[q] : i;   // LuT: x = P^T w
#pragma unroll
        for (int c = 0; c < RT; ++c)
          if (c0 + c < nrhs)
            Bs[idx(layouts >> 1, n, nrhs, srow, c0 + c) * ilv] = zero_x ? T(0) : b[q][c];
      }
    }
  }
}

template <typename T, int RT, int KIND, int Q, int WARPS>
cudaError_t launch_smem_q(int layout, int n, int nrhs, int64_t batch, const T* M,
                          const int32_t* ipiv, T* B, const int32_t* zinfo, cudaStream_t stream,
                          int64_t ilv) {
  const int64_t blocks = (batch + WARPS - 1) / WARPS;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const size_t bytes = static_cast<size_t>(WARPS) * n * odd_pitch(n) * sizeof(T);
  cudaError_t e = cudaFuncSetAttribute(solve_smem_kernel<T, RT, KIND, Q, WARPS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  solve_smem_kernel<T, RT, KIND, Q, WARPS><<<static_cast<unsigned>(blocks), WARPS * 32, bytes,
                                             stream>>>(n, nrhs, layout, batch, M, ipiv, B, zinfo,
                                                       ilv);
  return cudaGetLastError();
}

template <typename T, int KIND, int Q, int WARPS>
cudaError_t launch_smem_rhs(int layout, int n, int nrhs, int64_t batch, const T* M,
                            const int32_t* ipiv, T* B, const int32_t* zinfo,
                            cudaStream_t stream, int64_t ilv) {
  if (nrhs <= 1) return launch_smem_q<T, 1, KIND, Q, WARPS>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream, ilv);
  if (nrhs <= 2) return launch_smem_q<T, 2, KIND, Q, WARPS>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream, ilv);
  if (nrhs <= 4) return launch_smem_q<T, 4, KIND, Q, WARPS>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream, ilv);
  return launch_smem_q<T, 8, KIND, Q, WARPS>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream, ilv);
}

template <typename T, int KIND>
cudaError_t launch_smem(int layout, int n, int nrhs, int64_t batch, const T* M,
                        const int32_t* ipiv, T* B, const int32_t* zinfo, cudaStream_t stream,
                        int64_t ilv = 1) {
  if (n <= 64) return launch_smem_rhs<T, KIND, 2, 2>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream, ilv);
  return launch_smem_rhs<T, KIND, 4, 1>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream, ilv);
}

template <typename T, int KIND>
cudaError_t launch_kind(int layout, int n, int nrhs, int64_t batch, const T* M,
                        const int32_t* ipiv, T* B, const int32_t* zinfo, cudaStream_t stream) {
  if (n <= 4) return launch_reg_rhs<T, 4, 1, KIND>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream);
  if (n <= 8) return launch_reg_rhs<T, 8, kRows8, KIND>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream);
  if (n <= 16) return launch_reg_rhs<T, 16, kRows16, KIND>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream);
  if (n <= 32) return launch_reg_rhs<T, 32, kRows32, KIND>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream);
  if (n <= 128) return launch_smem<T, KIND>(layout, n, nrhs, batch, M, ipiv, B, zinfo, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

// `layout` of the launchers below is the packed code: bit 0 the storage order of the
// factor, bit 1 that of B (getrs: both the same; potrs with upper fill: the factor read as
// the lower triangle of the other order). zinfo (may be null): the factor's info, and X is
// written as zeros where it is not 0 (the fused calls' contract, when they run as a factor
// and a solve for more right-hand sides than a register tier holds).
// ilv > 1 (TDLS's interleaved batched layouts): one warp per system in shared memory for
// every n <= 128, the element offsets multiplied by the stride.
template <typename T>
cudaError_t launch_getrs(int layout, int n, int nrhs, int64_t batch, const T* LU,
                         const int32_t* ipiv, T* B, const int32_t* zinfo, cudaStream_t stream,
                         int64_t ilv) {
  if (ilv > 1) {
    if (n > 128) return cudaErrorInvalidValue;
    return launch_smem<T, kSolveLu>(layout, n, nrhs, batch, LU, ipiv, B, zinfo, stream, ilv);
  }
  return launch_kind<T, kSolveLu>(layout, n, nrhs, batch, LU, ipiv, B, zinfo, stream);
}

template <typename T>
cudaError_t launch_potrs(int layout, int n, int nrhs, int64_t batch, const T* L, T* B,
                         const int32_t* zinfo, cudaStream_t stream, int64_t ilv) {
  if (ilv > 1) {
    if (n > 128) return cudaErrorInvalidValue;
    return launch_smem<T, kSolveChol>(layout, n, nrhs, batch, L, nullptr, B, zinfo, stream, ilv);
  }
  // FP64, n <= 32, one right-hand side: one system per lane (solve_lane.cu)
  if constexpr (std::is_same<T, double>::value)
    if (n <= 32 && nrhs == 1) return launch_potrs_lane(layout, n, nrhs, batch, L, B, zinfo, stream);
  // orders beyond one CTA's shared memory: one CTA per system, the factor by tile columns
  if (n > 128) return launch_potrs_big(layout, n, nrhs, batch, L, B, zinfo, stream);
  return launch_kind<T, kSolveChol>(layout, n, nrhs, batch, L, nullptr, B, zinfo, stream);
}

template <typename T>
cudaError_t launch_getrs_mirror(int layout, int n, int nrhs, int64_t batch, const T* S,
                                const int32_t* ipiv, T* B, const int32_t* zinfo,
                                cudaStream_t stream, int64_t ilv) {
  if (ilv > 1) {
    if (n > 128) return cudaErrorInvalidValue;
    return launch_smem<T, kSolveLuT>(layout, n, nrhs, batch, S, ipiv, B, zinfo, stream, ilv);
  }
  return launch_kind<T, kSolveLuT>(layout, n, nrhs, batch, S, ipiv, B, zinfo, stream);
}

template cudaError_t launch_getrs<float>(int, int, int, int64_t, const float*, const int32_t*,
                                         float*, const int32_t*, cudaStream_t, int64_t);
template cudaError_t launch_getrs<double>(int, int, int, int64_t, const double*, const int32_t*,
                                          double*, const int32_t*, cudaStream_t, int64_t);
template cudaError_t launch_potrs<float>(int, int, int, int64_t, const float*, float*,
                                         const int32_t*, cudaStream_t, int64_t);
template cudaError_t launch_potrs<double>(int, int, int, int64_t, const double*, double*,
                                          const int32_t*, cudaStream_t, int64_t);
template cudaError_t launch_getrs_mirror<float>(int, int, int, int64_t, const float*,
                                                const int32_t*, float*, const int32_t*,
                                                cudaStream_t, int64_t);
template cudaError_t launch_getrs_mirror<double>(int, int, int, int64_t, const double*,
                                                 const int32_t*, double*, const int32_t*,
                                                 cudaStream_t, int64_t);

}  // namespace bsolve
