// LU with partial pivoting + solve for n <= 32, rows held in registers.
//
// One system per group of G = NT lanes (NT = the order tier, a power of two); 32/NT
// systems share a warp. Lane t holds physical row t of A and of B in registers for the
// whole solve, as in the TDLS CooperativeLUpp solver (TDLS API, "solver_static.hpp File
// Reference", Detailed Description): rows never move between lanes ("logical" row
// interchanges, MAGMA's rowid); each lane tracks the current position of its row.
//
// Step k (fully unrolled, every operand index static):
//   1. pivot search: live keys (the magnitude bits with the top bit set while the row is
//      still below the step, one OR per row; see LiveKey), the group max by one
//      full-warp redux.sync per group (FP32) or xor shuffles (FP64), then the lowest
//      current position among the lanes holding the max (lowest-row tie rule; a rare
//      exact tie takes a second reduction, a rare NaN candidate a rewrite of the keys);
//   2. positions k and p exchange (a bookkeeping swap, no data moves); the pivot lane
//      records the LAPACK swap entry ipiv[k] = position(p) + 1;
//   3. the pivot lane publishes its row (columns > k, from the 16-byte chunk holding
//      k+1, and the right-hand sides) with 16-byte stores in a shared-memory buffer,
//      double-buffered by step parity so that one __syncwarp per step orders writes and
//      reads;
//   4. every row still below the pivot scales its column-k entry by the pivot
//      reciprocal and applies the rank-1 update to its row of A and B (the forward solve
//      L y = P b folded into the factorization).
// Back substitution keeps x_i in the register of the lane that owns position i and
// publishes it through shared memory, one __syncwarp per step.
// Each row is written once, at its final position: the stored factor is in LAPACK
// order (row k = position k).
//
// Arithmetic (identical, operation by operation, to the CPU oracle): r = 1/pivot
// correctly rounded (r = 1 for a singular pivot), l = a_ik * r, every update one fused
// multiply-add, x_k = y_k * r_k.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace bsolve {
namespace lu_reg_detail {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;

template <typename T, int N>
__device__ __forceinline__ void load_vec(const T* __restrict__ p, T (&r)[N]) {
  if constexpr ((N * sizeof(T)) % 16 == 0) {
    constexpr int V = 16 / sizeof(T);
#pragma unroll
    for (int j = 0; j < N; j += V) {
      if constexpr (sizeof(T) == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p + j));
        r[j] = v.x; r[j + 1] = v.y; r[j + 2] = v.z; r[j + 3] = v.w;
      } else {
        const double2 v = __ldg(reinterpret_cast<const double2*>(p + j));
        r[j] = v.x; r[j + 1] = v.y;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) r[j] = p[j];
  }
}

template <typename T, int N>
__device__ __forceinline__ void store_vec(T* __restrict__ p, const T (&r)[N]) {
  if constexpr ((N * sizeof(T)) % 16 == 0) {
    constexpr int V = 16 / sizeof(T);
#pragma unroll
    for (int j = 0; j < N; j += V) {
      if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float4*>(p + j) = make_float4(r[j], r[j + 1], r[j + 2], r[j + 3]);
      } else {
        *reinterpret_cast<double2*>(p + j) = make_double2(r[j], r[j + 1]);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) p[j] = r[j];
  }
}

// Live pivot keys: the magnitude bits with the top bit set for a row still below the
// step and not yet a pivot row (0 otherwise). One OR per row orders |x| exactly, puts
// every live row above every dead or phantom one, and leaves the dead ones out of the tie
// rule. A live NaN has a key above inf's.
template <typename T> struct LiveKey;
template <> struct LiveKey<float> {
  using Key = uint32_t;
  static constexpr Key kAlive = 0x80000000u;
  static constexpr Key kNanAbove = 0xFF800000u;   // live key of inf
  static constexpr Key kRegular = 0x80800000u;    // live key of the smallest normal
  static constexpr Key kMax = 0xFFFFFFFFu;        // a NaN at the step's own position
  __device__ __forceinline__ static float value(Key k, unsigned sign) {
    return __uint_as_float((k & 0x7FFFFFFFu) | (sign << 31));
  }
};
template <> struct LiveKey<double> {
  using Key = unsigned long long;
  static constexpr Key kAlive = 0x8000000000000000ull;
  static constexpr Key kNanAbove = 0xFFF0000000000000ull;
  static constexpr Key kRegular = 0x8010000000000000ull;
  static constexpr Key kMax = 0xFFFFFFFFFFFFFFFFull;
  __device__ __forceinline__ static double value(Key k, unsigned sign) {
    return __longlong_as_double(static_cast<long long>(
        (k & 0x7FFFFFFFFFFFFFFFull) | (static_cast<unsigned long long>(sign) << 63)));
  }
};

// One 16-byte chunk of a register row to or from shared memory (j a multiple of 16/size).
template <typename T, int N>
__device__ __forceinline__ void st_chunk(T* p, const T (&r)[N], int j) {
  if constexpr (sizeof(T) == 4)
    *reinterpret_cast<float4*>(p) = make_float4(r[j], r[j + 1], r[j + 2], r[j + 3]);
  else
    *reinterpret_cast<double2*>(p) = make_double2(r[j], r[j + 1]);
}
template <typename T, int N>
__device__ __forceinline__ void ld_chunk(const T* p, T (&r)[N], int j) {
  if constexpr (sizeof(T) == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    r[j] = v.x; r[j + 1] = v.y; r[j + 2] = v.z; r[j + 3] = v.w;
  } else {
    const double2 v = *reinterpret_cast<const double2*>(p);
    r[j] = v.x; r[j + 1] = v.y;
  }
}
template <typename T, int N>
__device__ __forceinline__ void load_vec_shared(const T* p, T (&r)[N]) {
  if constexpr ((N * sizeof(T)) % 16 == 0) {
#pragma unroll
    for (int j = 0; j < N; j += 16 / sizeof(T)) ld_chunk<T, N>(p + j, r, j);
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) r[j] = p[j];
  }
}

// FULL: n == NT and nrhs == RT (every guard compiles away). RT = 0: factor only (getrf).
// IL: the interleaved batched layout (TDLS API, "solver_static.hpp File Reference":
// element e of system s at base_s[e * ilv], base_s = (s / ilv) * ilv * size + s % ilv,
// for A, B and ipiv; info one entry per system); ilv is read only when IL.
template <typename T, int NT, int RT, int LAYOUT, bool FULL, bool IL = false>
__global__ void __launch_bounds__(kThreads)
lu_reg_kernel(int n_, int nrhs_, int64_t batch, T* __restrict__ A, T* __restrict__ B,
              int32_t* __restrict__ ipiv, int32_t* __restrict__ info, int64_t ilv) {
  using Key = typename Traits<T>::Key;
  constexpr int G = NT;
  constexpr int GPW = 32 / G;                 // groups (systems) per warp
  constexpr bool kSolve = RT > 0;
  constexpr int RB = kSolve ? RT : 1;         // register / buffer size of the B part
  constexpr int W = NT + RT;                  // published row: A part, then B part
  constexpr int WP = (W * sizeof(T) + 15) / 16 * 16 / sizeof(T);
  constexpr unsigned GMASK = (G == 32) ? 0xFFFFFFFFu : ((1u << G) - 1u);

  __shared__ __align__(16) T prow[kWarps][GPW][2][WP];
  __shared__ __align__(16) T xbuf[kWarps][GPW][2][RB];
  // interleaved layout, staged: the block's systems (one AoSoA block holds them all) go
  // through shared memory with 16-byte accesses, each holding one element of VS systems;
  // row r of system j at (j*NT + r) * pitch (odd pitch: the lanes reading their rows hit
  // distinct banks)
  constexpr int SPC = kWarps * GPW;           // systems of a thread block
  constexpr int PA = NT + 1, PB = RB + 1;
  __shared__ __align__(16) T st_a[IL ? SPC * NT * PA : 1];
  __shared__ __align__(16) T st_b[IL ? SPC * NT * PB : 1];
  __shared__ __align__(16) int32_t st_p[IL ? SPC * NT : 1];

  const int n = FULL ? NT : n_;
  const int nrhs = FULL ? RT : nrhs_;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane / G;
  const int t = lane % G;
  const int64_t s = (static_cast<int64_t>(blockIdx.x) * kWarps + warp) * GPW + g;
  const bool valid = s < batch;
  const bool row_ok = valid && (FULL || t < n);

  T a[NT];
  T b[RB];
  const int64_t sA = s * n * n;
  const int64_t sB = s * n * nrhs;
  // interleaved: the system's first element of A, B and ipiv, and the element stride
  const int64_t blk = IL ? s / ilv : 0;
  const int64_t sl = IL ? s - blk * ilv : 0;
  const int64_t eA = IL ? blk * ilv * n * n + sl : 0;
  const int64_t eB = IL ? blk * ilv * n * nrhs + sl : 0;
  // staged when the block's systems fill whole 16-byte groups of one AoSoA block (the
  // last, partial thread block of a batch takes the scalar path): uniform per block
  const int64_t s_first = static_cast<int64_t>(blockIdx.x) * SPC;
  const bool staged = IL && ilv % SPC == 0 && s_first + SPC <= batch;
  const int jl = warp * GPW + g;                      // this group's system in the block
  constexpr int VS = 16 / sizeof(T);                 // elements of a 16-byte access
  const int64_t blk0 = IL ? s_first / ilv : 0;
  const int64_t sl0 = IL ? s_first - blk0 * ilv : 0;
  if (staged) {
    const T* const Ab = A + blk0 * ilv * n * n + sl0;
    const T* const Bb = B + blk0 * ilv * n * nrhs + sl0;
    constexpr int PER = SPC / VS;                      // vectors per element
    for (int idx = threadIdx.x; idx < n * n * PER; idx += kThreads) {
      const int e = idx / PER, q = idx - e * PER;
      const int r = LAYOUT == kRowMajor ? e / n : e % n;
      const int c = LAYOUT == kRowMajor ? e % n : e / n;
      T v[VS];
      ld_chunk<T, VS>(Ab + static_cast<int64_t>(e) * ilv + q * VS, v, 0);
#pragma unroll
      for (int u = 0; u < VS; ++u) st_a[((q * VS + u) * NT + r) * PA + c] = v[u];
    }
    if constexpr (kSolve) {
      for (int idx = threadIdx.x; idx < n * nrhs * PER; idx += kThreads) {
        const int e = idx / PER, q = idx - e * PER;
        const int r = LAYOUT == kRowMajor ? e / nrhs : e % n;
        const int c = LAYOUT == kRowMajor ? e % nrhs : e / n;
        T v[VS];
        ld_chunk<T, VS>(Bb + static_cast<int64_t>(e) * ilv + q * VS, v, 0);
#pragma unroll
        for (int u = 0; u < VS; ++u) st_b[((q * VS + u) * NT + r) * PB + c] = v[u];
      }
    }
    __syncthreads();
    if (row_ok) {
#pragma unroll
      for (int j = 0; j < NT; ++j) a[j] = j < n ? st_a[(jl * NT + t) * PA + j] : T(0);
#pragma unroll
      for (int c = 0; c < RB; ++c)
        b[c] = (kSolve && c < nrhs) ? st_b[(jl * NT + t) * PB + c] : T(0);
    } else {
#pragma unroll
      for (int j = 0; j < NT; ++j) a[j] = T(0);
#pragma unroll
      for (int c = 0; c < RB; ++c) b[c] = T(0);
    }
  } else if (IL && row_ok) {
#pragma unroll
    for (int j = 0; j < NT; ++j)
      a[j] = (FULL || j < n) ? A[eA + (LAYOUT == kRowMajor ? t * n + j : j * n + t) * ilv] : T(0);
#pragma unroll
    for (int c = 0; c < RT; ++c)
      b[c] = (FULL || c < nrhs)
                 ? B[eB + (LAYOUT == kRowMajor ? t * nrhs + c : c * n + t) * ilv] : T(0);
    if constexpr (!kSolve) b[0] = T(0);
  } else if (row_ok) {
    if (LAYOUT == kRowMajor) {
      if (FULL) {
        load_vec<T, NT>(A + sA + static_cast<int64_t>(t) * NT, a);
        if constexpr (kSolve) load_vec<T, RT>(B + sB + static_cast<int64_t>(t) * RT, b);
      } else {
#pragma unroll
        for (int j = 0; j < NT; ++j) a[j] = (j < n) ? A[sA + t * n + j] : T(0);
#pragma unroll
        for (int c = 0; c < RT; ++c) b[c] = (c < nrhs) ? B[sB + t * nrhs + c] : T(0);
        if constexpr (!kSolve) b[0] = T(0);
      }
    } else {
#pragma unroll
      for (int j = 0; j < NT; ++j) a[j] = (FULL || j < n) ? A[sA + j * n + t] : T(0);
#pragma unroll
      for (int c = 0; c < RT; ++c) b[c] = (FULL || c < nrhs) ? B[sB + c * n + t] : T(0);
      if constexpr (!kSolve) b[0] = T(0);
    }
  } else {
#pragma unroll
    for (int j = 0; j < NT; ++j) a[j] = T(0);
#pragma unroll
    for (int c = 0; c < RB; ++c) b[c] = T(0);
  }

  using LK = LiveKey<T>;
  Key alive = row_ok ? LK::kAlive : Key(0);   // live: below the step, not yet a pivot row
  int pos = t;          // current position of this lane's row
  int my_ipiv = 0;      // LAPACK entry of the step that chose this row
  T my_r = T(1);        // reciprocal of this row's pivot
  int inf = 0;
  constexpr int V = 16 / sizeof(T);

  // the group maximum of a key: one full-warp redux.sync per group for FP32 (non-members
  // contribute 0, below every key; shorter latency than a shuffle butterfly and cheaper
  // than a partial-mask redux), xor shuffles for FP64
  auto group_max = [&](Key key) {
    Key mk;
    if constexpr (sizeof(Key) == 4 && GPW <= 4) {
      mk = 0;
#pragma unroll
      for (int q = 0; q < GPW; ++q) {
        const Key m = __reduce_max_sync(0xFFFFFFFFu, g == q ? key : Key(0));
        mk = (g == q) ? m : mk;
      }
    } else {
      mk = key;
#pragma unroll
      for (int off = G / 2; off >= 1; off >>= 1) {
        const Key o = shfl_xor_key(mk, off, G);
        mk = o > mk ? o : mk;
      }
    }
    return mk;
  };

#pragma unroll
  for (int k = 0; k < NT; ++k) {
    if (!FULL && k >= n) break;
    Key key = Traits<T>::mag_bits(a[k]) | alive;
    Key mk = group_max(key);
    if (__any_sync(0xFFFFFFFFu, mk > LK::kNanAbove)) {
      // a NaN among some group's candidates (rare): the contract's keys, a NaN at the
      // step's own position wins, a NaN elsewhere ties with zero
      if (key > LK::kNanAbove) key = (pos == k) ? LK::kMax : LK::kAlive;
      mk = group_max(key);
    }
    const unsigned sbal = __ballot_sync(0xFFFFFFFFu, signbit(a[k]));
    const bool hold = key == mk;
    const unsigned bal = (__ballot_sync(0xFFFFFFFFu, hold) >> (g * G)) & GMASK;
    int plane;
    if (__any_sync(0xFFFFFFFFu, __popc(bal) > 1)) {
      // exact tie: the lowest current position among the lanes holding the max
      int tp = hold ? pos : 0x7FFFFFFF;
#pragma unroll
      for (int off = G / 2; off >= 1; off >>= 1) {
        const int o = __shfl_xor_sync(0xFFFFFFFFu, tp, off, G);
        tp = o < tp ? o : tp;
      }
      const unsigned b2 =
          (__ballot_sync(0xFFFFFFFFu, hold && pos == tp) >> (g * G)) & GMASK;
      plane = __ffs(b2) - 1;
    } else {
      plane = __ffs(bal) - 1;
    }
    if (plane < 0) plane = 0;  // only in groups past the end of the batch
    const int pos_p = __shfl_sync(0xFFFFFFFFu, pos, plane, G);
    const bool ok = mk >= LK::kRegular && mk != LK::kMax;
    if (!ok && inf == 0) inf = k + 1;
    const bool is_p = (t == plane);
    if (pos == k) pos = pos_p;
    if (is_p) {
      my_ipiv = pos_p + 1;
      pos = k;
      alive = 0;
    }

    // The pivot is known without waiting for the published row: its magnitude is in the
    // max key, its sign the pivot lane's bit of the sign ballot. The reciprocal and the
    // multipliers thus overlap the shared-memory round trip of the pivot row.
    const T piv = LK::value(mk, (sbal >> (g * G + plane)) & 1u);
    const T r = ok ? T(1) / piv : T(1);
    if (is_p) my_r = r;
    const bool upd = alive != 0;
    const T l = a[k] * r;
    if (upd) a[k] = l;

    // the pivot row's columns > k (from the 16-byte chunk holding k+1) and its B part
    T* pr = prow[warp][g][k & 1];
    const int c1 = (k + 1) & ~(V - 1);
    if (is_p) {
#pragma unroll
      for (int j = 0; j < NT; j += V)
        if (j >= c1) st_chunk<T>(pr + j, a, j);
      if constexpr (kSolve) store_vec<T, RT>(pr + NT, b);
    }
    __syncwarp();
    if (upd) {
      T u[NT];
#pragma unroll
      for (int j = 0; j < NT; j += V)
        if (j >= c1) ld_chunk<T>(pr + j, u, j);
      T ub[RB];
      if constexpr (kSolve) load_vec_shared<T, RT>(pr + NT, ub);
#pragma unroll
      for (int j = k + 1; j < NT; ++j) a[j] = fma_rn<T>(-l, u[j], a[j]);
#pragma unroll
      for (int c = 0; c < RT; ++c) b[c] = fma_rn<T>(-l, ub[c], b[c]);
    }
  }

  // U x = y, from the last position.
#pragma unroll
  for (int i = NT - 1; i >= 0; --i) {
    if constexpr (!kSolve) break;
    if (!FULL && i >= n) continue;
    T* xb = xbuf[warp][g][i & 1];
    if (row_ok && pos == i) {
#pragma unroll
      for (int c = 0; c < RT; ++c) {
        b[c] = b[c] * my_r;
        xb[c] = b[c];
      }
    }
    __syncwarp();
    if (row_ok && pos < i) {
#pragma unroll
      for (int c = 0; c < RT; ++c) b[c] = fma_rn<T>(-a[i], xb[c], b[c]);
    }
  }

  if (staged) {
    if (row_ok) {
      if (inf != 0) {
#pragma unroll
        for (int c = 0; c < RT; ++c) b[c] = T(0);
      }
#pragma unroll
      for (int j = 0; j < NT; ++j)
        if (j < n) st_a[(jl * NT + pos) * PA + j] = a[j];
#pragma unroll
      for (int c = 0; c < RT; ++c)
        if (c < nrhs) st_b[(jl * NT + pos) * PB + c] = b[c];
      st_p[jl * NT + pos] = my_ipiv;
      if (t == 0) info[s] = inf;
    }
    __syncthreads();
    T* const Ab = A + blk0 * ilv * n * n + sl0;
    T* const Bb = B + blk0 * ilv * n * nrhs + sl0;
    int32_t* const Pb = ipiv + blk0 * ilv * n + sl0;
    constexpr int PER = SPC / VS;
    for (int idx = threadIdx.x; idx < n * n * PER; idx += kThreads) {
      const int e = idx / PER, q = idx - e * PER;
      const int r = LAYOUT == kRowMajor ? e / n : e % n;
      const int c = LAYOUT == kRowMajor ? e % n : e / n;
      T v[VS];
#pragma unroll
      for (int u = 0; u < VS; ++u) v[u] = st_a[((q * VS + u) * NT + r) * PA + c];
      st_chunk<T, VS>(Ab + static_cast<int64_t>(e) * ilv + q * VS, v, 0);
    }
    if constexpr (kSolve) {
      for (int idx = threadIdx.x; idx < n * nrhs * PER; idx += kThreads) {
        const int e = idx / PER, q = idx - e * PER;
        const int r = LAYOUT == kRowMajor ? e / nrhs : e % n;
        const int c = LAYOUT == kRowMajor ? e % nrhs : e / n;
        T v[VS];
#pragma unroll
        for (int u = 0; u < VS; ++u) v[u] = st_b[((q * VS + u) * NT + r) * PB + c];
        st_chunk<T, VS>(Bb + static_cast<int64_t>(e) * ilv + q * VS, v, 0);
      }
    }
    constexpr int PERI = SPC / 4;                     // ipiv: four systems per 16 bytes
    for (int idx = threadIdx.x; idx < n * PERI; idx += kThreads) {
      const int k = idx / PERI, q = idx - k * PERI;
      *reinterpret_cast<int4*>(Pb + static_cast<int64_t>(k) * ilv + q * 4) =
          make_int4(st_p[(q * 4) * NT + k], st_p[(q * 4 + 1) * NT + k],
                    st_p[(q * 4 + 2) * NT + k], st_p[(q * 4 + 3) * NT + k]);
    }
  } else if (IL && row_ok) {
    if (inf != 0) {
#pragma unroll
      for (int c = 0; c < RT; ++c) b[c] = T(0);
    }
#pragma unroll
    for (int j = 0; j < NT; ++j)
      if (FULL || j < n) A[eA + (LAYOUT == kRowMajor ? pos * n + j : j * n + pos) * ilv] = a[j];
#pragma unroll
    for (int c = 0; c < RT; ++c)
      if (FULL || c < nrhs) B[eB + (LAYOUT == kRowMajor ? pos * nrhs + c : c * n + pos) * ilv] = b[c];
    ipiv[blk * ilv * n + sl + pos * ilv] = my_ipiv;
    if (t == 0) info[s] = inf;
  } else if (row_ok) {
    if (inf != 0) {
#pragma unroll
      for (int c = 0; c < RT; ++c) b[c] = T(0);
    }
    if (LAYOUT == kRowMajor) {
      if (FULL) {
        store_vec<T, NT>(A + sA + static_cast<int64_t>(pos) * NT, a);
        if constexpr (kSolve) store_vec<T, RT>(B + sB + static_cast<int64_t>(pos) * RT, b);
      } else {
#pragma unroll
        for (int j = 0; j < NT; ++j)
          if (j < n) A[sA + pos * n + j] = a[j];
#pragma unroll
        for (int c = 0; c < RT; ++c)
          if (c < nrhs) B[sB + pos * nrhs + c] = b[c];
      }
    } else {
#pragma unroll
      for (int j = 0; j < NT; ++j)
        if (FULL || j < n) A[sA + j * n + pos] = a[j];
#pragma unroll
      for (int c = 0; c < RT; ++c)
        if (FULL || c < nrhs) B[sB + c * n + pos] = b[c];
    }
    ipiv[s * n + pos] = my_ipiv;
    if (t == 0) info[s] = inf;
  }
}

template <typename T, int NT, int RT, int LAYOUT>
cudaError_t launch_tier(int n, int nrhs, int64_t batch, T* A, T* B, int32_t* ipiv,
                        int32_t* info, cudaStream_t stream) {
  constexpr int per_block = kWarps * (32 / NT);
  const int64_t blocks = (batch + per_block - 1) / per_block;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  if (n == NT && nrhs == RT)
    lu_reg_kernel<T, NT, RT, LAYOUT, true><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        n, nrhs, batch, A, B, ipiv, info, 1);
  else
    lu_reg_kernel<T, NT, RT, LAYOUT, false><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        n, nrhs, batch, A, B, ipiv, info, 1);
  return cudaGetLastError();
}

// The interleaved batched layout, systems in blocks of ilv: per tier an instance without
// guards (n and nrhs the tier's) and one with them.
template <typename T, int NT, int RT, int LAYOUT>
cudaError_t launch_tier_il(int n, int nrhs, int64_t batch, int64_t ilv, T* A, T* B,
                           int32_t* ipiv, int32_t* info, cudaStream_t stream) {
  constexpr int per_block = kWarps * (32 / NT);
  const int64_t blocks = (batch + per_block - 1) / per_block;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  if (n == NT && nrhs == RT)   // the order and right-hand sides of the tier: no guards
    lu_reg_kernel<T, NT, RT, LAYOUT, true, true>
        <<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(n, nrhs, batch, A, B, ipiv,
                                                                 info, ilv);
  else
    lu_reg_kernel<T, NT, RT, LAYOUT, false, true>
        <<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(n, nrhs, batch, A, B, ipiv,
                                                                 info, ilv);
  return cudaGetLastError();
}

template <typename T, int NT, int LAYOUT>
cudaError_t launch_rhs_il(int n, int nrhs, int64_t batch, int64_t ilv, T* A, T* B,
                          int32_t* ipiv, int32_t* info, cudaStream_t stream) {
  if (nrhs <= 1) return launch_tier_il<T, NT, 1, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  if (nrhs <= 2) return launch_tier_il<T, NT, 2, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  if (nrhs <= 4) return launch_tier_il<T, NT, 4, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  return launch_tier_il<T, NT, 8, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
}

template <typename T, int LAYOUT>
cudaError_t launch_layout_il(int n, int nrhs, int64_t batch, int64_t ilv, T* A, T* B,
                             int32_t* ipiv, int32_t* info, cudaStream_t stream) {
  if (n <= 4) return launch_rhs_il<T, 4, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  if (n <= 8) return launch_rhs_il<T, 8, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  if (n <= 16) return launch_rhs_il<T, 16, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  return launch_rhs_il<T, 32, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
}

template <typename T, int NT, int LAYOUT>
cudaError_t launch_rhs(int n, int nrhs, int64_t batch, T* A, T* B, int32_t* ipiv, int32_t* info,
                       cudaStream_t stream) {
  if (nrhs == 0) return launch_tier<T, NT, 0, LAYOUT>(n, nrhs, batch, A, B, ipiv, info, stream);
  if (nrhs <= 1) return launch_tier<T, NT, 1, LAYOUT>(n, nrhs, batch, A, B, ipiv, info, stream);
  if (nrhs <= 2) return launch_tier<T, NT, 2, LAYOUT>(n, nrhs, batch, A, B, ipiv, info, stream);
  if (nrhs <= 4) return launch_tier<T, NT, 4, LAYOUT>(n, nrhs, batch, A, B, ipiv, info, stream);
  return launch_tier<T, NT, 8, LAYOUT>(n, nrhs, batch, A, B, ipiv, info, stream);
}

template <typename T, int LAYOUT>
cudaError_t launch_layout(int n, int nrhs, int64_t batch, T* A, T* B, int32_t* ipiv,
                          int32_t* info, cudaStream_t stream) {
  if (n <= 4) return launch_rhs<T, 4, LAYOUT>(n, nrhs, batch, A, B, ipiv, info, stream);
  if (n <= 8) return launch_rhs<T, 8, LAYOUT>(n, nrhs, batch, A, B, ipiv, info, stream);
  if (n <= 16) return launch_rhs<T, 16, LAYOUT>(n, nrhs, batch, A, B, ipiv, info, stream);
  return launch_rhs<T, 32, LAYOUT>(n, nrhs, batch, A, B, ipiv, info, stream);
}

}  // namespace lu_reg_detail
}  // namespace bsolve
