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

constexpr int kThreads = 128;

template <int BS>
struct Tri {
  static constexpr int kSize = BS * (BS + 1) / 2;
  __host__ __device__ static constexpr int at(int i, int j) { return i * (i + 1) / 2 + j; }
};

// MODE: kFused (factor + solve, the forward solve riding on the factor sweep),
// kFactor (strips only), kSolve (strips already factored, read only).
enum Mode : int { kFused = 0, kFactor = 1, kSolve = 2 };

template <typename T, int BS, int MODE>
__global__ void __launch_bounds__(kThreads)
bdsv_kernel(int nbr, int64_t batch, T* __restrict__ strips, T* __restrict__ xpad,
            int32_t* __restrict__ info) {
  constexpr int W = 3 * BS;
  constexpr bool kFactors = MODE != kSolve;   // computes F_k, E_k
  constexpr bool kSolves = MODE != kFactor;   // computes y, x
  using Tr = Tri<BS>;
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
    if constexpr (kSolves) {
#pragma unroll
      for (int i = 0; i < BS; ++i) z[i] = x[k * BS + i];
    }
    if constexpr (kFactors) {
#pragma unroll
      for (int i = 0; i < BS; ++i)
#pragma unroll
        for (int j = 0; j <= i; ++j) Sm[Tr::at(i, j)] = strip[i * W + BS + j];
    }
    if (k > 0) {
      T E[BS][BS];
      if constexpr (kFactors) {
        // E_k = L_k F_{k-1}^{-T}, row by row
#pragma unroll
        for (int a = 0; a < BS; ++a) {
#pragma unroll
          for (int j = 0; j < BS; ++j) {
            T acc = strip[a * W + j];
#pragma unroll
            for (int m = 0; m < j; ++m) acc = fma_rn<T>(-E[a][m], F[Tr::at(j, m)], acc);
            E[a][j] = acc * Fr[j];
          }
        }
#pragma unroll
        for (int a = 0; a < BS; ++a)
#pragma unroll
          for (int j = 0; j < BS; ++j) strip[a * W + j] = E[a][j];
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
        for (int a = 0; a < BS; ++a)
#pragma unroll
          for (int j = 0; j < BS; ++j) E[a][j] = strip[a * W + j];
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
        if (!failed && !(d > T(0))) {
          failed = true;
          inf = k * BS + c + 1;
        }
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
      for (int i = 0; i < BS; ++i)
#pragma unroll
        for (int j = 0; j <= i; ++j) strip[i * W + BS + j] = Sm[Tr::at(i, j)];
    } else {
#pragma unroll
      for (int i = 0; i < BS; ++i)
#pragma unroll
        for (int j = 0; j <= i; ++j) Sm[Tr::at(i, j)] = strip[i * W + BS + j];
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
#pragma unroll
      for (int j = 0; j < BS; ++j) x[k * BS + j] = y[j];
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
#pragma unroll
      for (int i = 0; i < BS; ++i) w[i] = x[k * BS + i];
      if (k < nbr - 1) {
        const T* nstrip = strip + BS * W;
#pragma unroll
        for (int m = 0; m < BS; ++m)
#pragma unroll
          for (int i = 0; i < BS; ++i) w[m] = fma_rn<T>(-nstrip[i * W + m], xn[i], w[m]);
      }
#pragma unroll
      for (int i = 0; i < BS; ++i)
#pragma unroll
        for (int j = 0; j <= i; ++j) F[Tr::at(i, j)] = strip[i * W + BS + j];
      T xk[BS];
#pragma unroll
      for (int j = BS - 1; j >= 0; --j) {
        T acc = w[j];
#pragma unroll
        for (int m = j + 1; m < BS; ++m) acc = fma_rn<T>(-F[Tr::at(m, j)], xk[m], acc);
        xk[j] = acc * rcp_rn<T>(F[Tr::at(j, j)]);
      }
#pragma unroll
      for (int j = 0; j < BS; ++j) {
        x[k * BS + j] = xk[j];
        xn[j] = xk[j];
      }
    }
    if (MODE == kFused) info[s] = 0;
  }
}

template <typename T, int BS, int MODE>
cudaError_t launch_bs(int nbr, int64_t batch, T* strips, T* xpad, int32_t* info,
                      cudaStream_t stream) {
  const int64_t blocks = (batch + kThreads - 1) / kThreads;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  bdsv_kernel<T, BS, MODE><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
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
