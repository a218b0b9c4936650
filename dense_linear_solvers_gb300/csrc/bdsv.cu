// Block-tridiagonal SPD solve by the block-Cholesky (block-Thomas) sweep, one thread
// per system (GLASS API reference, "Block-tridiagonal Ops", section "Direct solve
// (glass::bdsv)"): F_0 = chol(D_0); E_k = L_k F_{k-1}^{-T}; F_k = chol(D_k - E_k E_k^T);
// y_k = F_k^{-1}(b_k - E_k y_{k-1}); x_k = F_k^{-T}(y_k - E_{k+1}^T x_{k+1}).
//
// The chain over knots is serial; GLASS spreads each knot's small BLAS over a thread
// block. Here every lane of a warp runs the whole sweep of its own system with the
// block size BS a compile-time constant, so every floating-point instruction of the
// warp does useful work on 32 systems at once (on a part whose FP64 pipe charges a
// warp instruction whatever its active lanes, idle lanes inside a knot would be paid
// for). Strips are read and written in place, rows of 16 bytes at a time; the factor
// written in the forward sweep is read back in the backward sweep.
// The same kernel runs the fused solve (bdsv), the factor sweep alone (bdsv_factor: MAIN
// <- F_k, LEFT <- E_k, info) and the substitutions alone on factored strips (bdsv_solve,
// strips read only, the diagonal reciprocals recomputed: "factor once, call this per
// right-hand side").
// The arithmetic is the CPU oracle's, operation by operation.
#include "common.cuh"
#include "kernels.h"

namespace bsolve {
namespace {

constexpr int kThreads = 32;

template <int BS>
struct Tri {
  static constexpr int kSize = BS * (BS + 1) / 2;
  __host__ __device__ static constexpr int at(int i, int j) { return i * (i + 1) / 2 + j; }
};

// n contiguous elements at p to d (or d to p): 32-byte pieces where whole when W32 (FP64,
// strips and x 32-byte aligned), then 16-byte pieces when VEC (the address then 16-byte
// aligned by construction), the rest element by element; nothing at or past p[n] is
// touched.
struct __align__(32) D4 {
  double v[4];
};

template <typename T, bool VEC, bool W32>
__device__ __forceinline__ void ld_n(const T* p, T* d, int n) {
  constexpr int VW = 16 / sizeof(T);
  const int n32 = (W32 && sizeof(T) == 8) ? n / 4 : 0;   // 32-byte pieces (FP64)
  const int nv = VEC ? (n - 4 * n32) / VW : 0;
#pragma unroll
  for (int q = 0; q < n32; ++q) {
    const D4 v = reinterpret_cast<const D4*>(p)[q];
    double* o = reinterpret_cast<double*>(d) + 4 * q;
    o[0] = v.v[0]; o[1] = v.v[1]; o[2] = v.v[2]; o[3] = v.v[3];
  }
  const T* pv = p + 4 * n32;
  T* dv = d + 4 * n32;
#pragma unroll
  for (int q = 0; q < nv; ++q) {
    if constexpr (sizeof(T) == 8) {
      const double2 v = *reinterpret_cast<const double2*>(pv + q * VW);
      dv[q * VW] = v.x; dv[q * VW + 1] = v.y;
    } else {
      const float4 v = *reinterpret_cast<const float4*>(pv + q * VW);
      dv[q * VW] = v.x; dv[q * VW + 1] = v.y; dv[q * VW + 2] = v.z; dv[q * VW + 3] = v.w;
    }
  }
#pragma unroll
  for (int j = 4 * n32 + nv * VW; j < n; ++j) d[j] = p[j];
}
template <typename T, bool VEC, bool W32>
__device__ __forceinline__ void st_n(T* p, const T* d, int n) {
  constexpr int VW = 16 / sizeof(T);
  const int n32 = (W32 && sizeof(T) == 8) ? n / 4 : 0;
  const int nv = VEC ? (n - 4 * n32) / VW : 0;
#pragma unroll
  for (int q = 0; q < n32; ++q) {
    const double* o = reinterpret_cast<const double*>(d) + 4 * q;
    D4 v;
    v.v[0] = o[0]; v.v[1] = o[1]; v.v[2] = o[2]; v.v[3] = o[3];
    reinterpret_cast<D4*>(p)[q] = v;
  }
  T* pv = p + 4 * n32;
  const T* dv = d + 4 * n32;
#pragma unroll
  for (int q = 0; q < nv; ++q) {
    if constexpr (sizeof(T) == 8)
      *reinterpret_cast<double2*>(pv + q * VW) = make_double2(dv[q * VW], dv[q * VW + 1]);
    else
      *reinterpret_cast<float4*>(pv + q * VW) =
          make_float4(dv[q * VW], dv[q * VW + 1], dv[q * VW + 2], dv[q * VW + 3]);
  }
#pragma unroll
  for (int j = 4 * n32 + nv * VW; j < n; ++j) p[j] = d[j];
}

// MODE: kFused (factor + solve, the forward solve riding on the factor sweep),
// kFactor (strips only), kSolve (strips already factored, read only).
enum Mode : int { kFused = 0, kFactor = 1, kSolve = 2 };

template <typename T, int BS, int MODE, bool W32>
__global__ void __launch_bounds__(kThreads)
bdsv_kernel(int nbr, int64_t batch, T* __restrict__ strips, T* __restrict__ xpad,
            int32_t* __restrict__ info) {
  constexpr int W = 3 * BS;
  constexpr bool kFactors = MODE != kSolve;   // computes F_k, E_k
  constexpr bool kSolves = MODE != kFactor;   // computes y, x
  using Tr = Tri<BS>;
  // every row of a strip, the diagonal block's columns and every block of x start on a
  // 16-byte boundary when a block row is a whole number of 16-byte pieces (the bases are
  // 16-byte aligned)
  constexpr bool VEC = (BS * sizeof(T)) % 16 == 0;
  const int64_t s = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (s >= batch) return;
  T* S = strips + s * static_cast<int64_t>(nbr) * BS * W;
  T* x = xpad + s * static_cast<int64_t>(nbr + 2) * BS + BS;

  T F[Tr::kSize];   // F_{k-1} (factoring) or F_k (solving), lower, packed by rows
  T Fr[BS];         // reciprocals of its diagonal
  T y[BS];          // y_{k-1}
#pragma unroll
  for (int i = 0; i < BS; ++i) y[i] = T(0);
  int inf = 0;

  for (int k = 0; k < nbr; ++k) {
    T* strip = S + static_cast<int64_t>(k) * BS * W;
    T Sm[Tr::kSize];
    T z[BS];
    if constexpr (kSolves) ld_n<T, VEC, W32>(x + k * BS, z, BS);
    // D_k's lower triangle (at the knot's start for k = 0, after E_k otherwise: fewer live
    // registers while E_k is formed)
    if constexpr (kFactors) {
      if (k == 0) {
#pragma unroll
        for (int i = 0; i < BS; ++i) ld_n<T, VEC, W32>(strip + i * W + BS, &Sm[Tr::at(i, 0)], i + 1);
      }
    }
    if (k > 0) {
      T E[BS][BS];
      if constexpr (kFactors) {
        // E_k = L_k F_{k-1}^{-T}, row by row
#pragma unroll
        for (int a = 0; a < BS; ++a) {
          T Lrow[BS];
          ld_n<T, VEC, W32>(strip + a * W, Lrow, BS);
#pragma unroll
          for (int j = 0; j < BS; ++j) {
            T acc = Lrow[j];
#pragma unroll
            for (int m = 0; m < j; ++m) acc = fma_rn<T>(-E[a][m], F[Tr::at(j, m)], acc);
            E[a][j] = acc * Fr[j];
          }
        }
#pragma unroll
        for (int a = 0; a < BS; ++a) st_n<T, VEC, W32>(strip + a * W, E[a], BS);
#pragma unroll
        for (int i = 0; i < BS; ++i) ld_n<T, VEC, W32>(strip + i * W + BS, &Sm[Tr::at(i, 0)], i + 1);
        // S_k = D_k - E_k E_k^T (lower)
#pragma unroll
        for (int i = 0; i < BS; ++i)
#pragma unroll
          for (int j = 0; j <= i; ++j) {
            T acc = Sm[Tr::at(i, j)];
#pragma unroll
            for (int m = 0; m < BS; ++m) acc = fma_rn<T>(-E[i][m], E[j][m], acc);
            Sm[Tr::at(i, j)] = acc;
          }
      } else {
#pragma unroll
        for (int a = 0; a < BS; ++a) ld_n<T, VEC, W32>(strip + a * W, E[a], BS);
      }
      if constexpr (kSolves) {
#pragma unroll
        for (int i = 0; i < BS; ++i)
#pragma unroll
          for (int m = 0; m < BS; ++m) z[i] = fma_rn<T>(-E[i][m], y[m], z[i]);
      }
    }
    if constexpr (kFactors) {
      // F_k = chol(S_k), right-looking
      bool failed = false;
#pragma unroll
      for (int c = 0; c < BS; ++c) {
        const T d = Sm[Tr::at(c, c)];
        // branch-free, so that the whole knot stays one block of straight-line code and
        // the compiler can overlap one column's square root and reciprocal with the
        // previous column's independent updates
        const bool bad = !(d > T(0));
        inf = (!failed && bad) ? k * BS + c + 1 : inf;
        failed = failed || bad;
        const T l = sqrt_rn<T>(d);
        const T r = rcp_rn<T>(l);
        Sm[Tr::at(c, c)] = l;
        Fr[c] = r;
#pragma unroll
        for (int i = c + 1; i < BS; ++i) Sm[Tr::at(i, c)] = Sm[Tr::at(i, c)] * r;
#pragma unroll
        for (int j = c + 1; j < BS; ++j) {
          const T ljc = Sm[Tr::at(j, c)];
#pragma unroll
          for (int i = j; i < BS; ++i)
            Sm[Tr::at(i, j)] = fma_rn<T>(-Sm[Tr::at(i, c)], ljc, Sm[Tr::at(i, j)]);
        }
      }
      if (failed) break;
#pragma unroll
      for (int i = 0; i < BS; ++i) st_n<T, VEC, W32>(strip + i * W + BS, &Sm[Tr::at(i, 0)], i + 1);
    } else {
#pragma unroll
      for (int i = 0; i < BS; ++i) ld_n<T, VEC, W32>(strip + i * W + BS, &Sm[Tr::at(i, 0)], i + 1);
#pragma unroll
      for (int c = 0; c < BS; ++c) Fr[c] = rcp_rn<T>(Sm[Tr::at(c, c)]);
    }
    if constexpr (kSolves) {
      // y_k = F_k^{-1} z
#pragma unroll
      for (int j = 0; j < BS; ++j) {
        T acc = z[j];
#pragma unroll
        for (int m = 0; m < j; ++m) acc = fma_rn<T>(-Sm[Tr::at(j, m)], y[m], acc);
        y[j] = acc * Fr[j];
      }
      st_n<T, VEC, W32>(x + k * BS, y, BS);
    }
    if constexpr (kFactors) {
#pragma unroll
      for (int e = 0; e < Tr::kSize; ++e) F[e] = Sm[e];
    }
  }

  if constexpr (!kSolves) {
    info[s] = inf;
    return;
  } else {
    if (inf != 0) {
      for (int i = 0; i < nbr * BS; ++i) x[i] = T(0);
      info[s] = inf;
      return;
    }
    // backward sweep: x_k = F_k^{-T}(y_k - E_{k+1}^T x_{k+1})
    T xn[BS];
    for (int k = nbr - 1; k >= 0; --k) {
      const T* strip = S + static_cast<int64_t>(k) * BS * W;
      T w[BS];
      ld_n<T, VEC, W32>(x + k * BS, w, BS);
      if (k < nbr - 1) {
        // each w[m] takes its updates in increasing i, row i of E_{k+1} at a time
        const T* nstrip = strip + BS * W;
#pragma unroll
        for (int i = 0; i < BS; ++i) {
          T er[BS];
          ld_n<T, VEC, W32>(nstrip + i * W, er, BS);
#pragma unroll
          for (int m = 0; m < BS; ++m) w[m] = fma_rn<T>(-er[m], xn[i], w[m]);
        }
      }
#pragma unroll
      for (int i = 0; i < BS; ++i) ld_n<T, VEC, W32>(strip + i * W + BS, &F[Tr::at(i, 0)], i + 1);
      T xk[BS];
#pragma unroll
      for (int j = BS - 1; j >= 0; --j) {
        T acc = w[j];
#pragma unroll
        for (int m = j + 1; m < BS; ++m) acc = fma_rn<T>(-F[Tr::at(m, j)], xk[m], acc);
        xk[j] = acc * rcp_rn<T>(F[Tr::at(j, j)]);
      }
      st_n<T, VEC, W32>(x + k * BS, xk, BS);
#pragma unroll
      for (int j = 0; j < BS; ++j) xn[j] = xk[j];
    }
    if (MODE == kFused) info[s] = 0;
  }
}

template <typename T, int BS, int MODE>
cudaError_t launch_bs(int nbr, int64_t batch, T* strips, T* xpad, int32_t* info,
                      cudaStream_t stream) {
  const int64_t blocks = (batch + kThreads - 1) / kThreads;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  // 32-byte accesses for FP64 block rows of whole 32-byte pieces when both bases allow
  const bool w32 = sizeof(T) == 8 && (BS * sizeof(T)) % 32 == 0 &&
                   reinterpret_cast<uintptr_t>(strips) % 32 == 0 &&
                   (xpad == nullptr || reinterpret_cast<uintptr_t>(xpad) % 32 == 0);
  if (w32)
    bdsv_kernel<T, BS, MODE, true><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        nbr, batch, strips, xpad, info);
  else
    bdsv_kernel<T, BS, MODE, false><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        nbr, batch, strips, xpad, info);
  return cudaGetLastError();
}

template <typename T, int MODE>
cudaError_t launch_mode(int nbr, int bs, int64_t batch, T* strips, T* xpad, int32_t* info,
                        cudaStream_t stream) {
  switch (bs) {
    case 1: return launch_bs<T, 1, MODE>(nbr, batch, strips, xpad, info, stream);
    case 2: return launch_bs<T, 2, MODE>(nbr, batch, strips, xpad, info, stream);
    case 3: return launch_bs<T, 3, MODE>(nbr, batch, strips, xpad, info, stream);
    case 4: return launch_bs<T, 4, MODE>(nbr, batch, strips, xpad, info, stream);
    case 5: return launch_bs<T, 5, MODE>(nbr, batch, strips, xpad, info, stream);
    case 6: return launch_bs<T, 6, MODE>(nbr, batch, strips, xpad, info, stream);
    case 7: return launch_bs<T, 7, MODE>(nbr, batch, strips, xpad, info, stream);
    case 8: return launch_bs<T, 8, MODE>(nbr, batch, strips, xpad, info, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

template <typename T>
cudaError_t launch_bdsv(int nbr, int bs, int64_t batch, T* strips, T* xpad, int32_t* info,
                        cudaStream_t stream) {
  return launch_mode<T, kFused>(nbr, bs, batch, strips, xpad, info, stream);
}

template <typename T>
cudaError_t launch_bdsv_factor(int nbr, int bs, int64_t batch, T* strips, int32_t* info,
                               cudaStream_t stream) {
  return launch_mode<T, kFactor>(nbr, bs, batch, strips, nullptr, info, stream);
}

template <typename T>
cudaError_t launch_bdsv_solve(int nbr, int bs, int64_t batch, const T* strips, T* xpad,
                              cudaStream_t stream) {
  // the solve only reads the strips
  return launch_mode<T, kSolve>(nbr, bs, batch, const_cast<T*>(strips), xpad, nullptr, stream);
}

template cudaError_t launch_bdsv<float>(int, int, int64_t, float*, float*, int32_t*,
                                        cudaStream_t);
template cudaError_t launch_bdsv<double>(int, int, int64_t, double*, double*, int32_t*,
                                         cudaStream_t);
template cudaError_t launch_bdsv_factor<float>(int, int, int64_t, float*, int32_t*, cudaStream_t);
template cudaError_t launch_bdsv_factor<double>(int, int, int64_t, double*, int32_t*,
                                                cudaStream_t);
template cudaError_t launch_bdsv_solve<float>(int, int, int64_t, const float*, float*,
                                              cudaStream_t);
template cudaError_t launch_bdsv_solve<double>(int, int, int64_t, const double*, double*,
                                               cudaStream_t);

}  // namespace bsolve
