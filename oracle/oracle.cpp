// Sequential CPU oracle for the batched small dense solvers.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls this
// file: only the test suite, the smoke check and the benchmark's CPU-baseline leg do.
// It shares no source, header, table or helper with the CUDA library.
//
// Every routine solves one system at a time, in the arithmetic type of its inputs
// (float or double), with the textbook operation order written out below. The batch
// loops only hand whole systems to worker threads; the arithmetic of a system never
// depends on the thread count.
//
// Arithmetic convention shared by every routine (where the pages leave rounding open):
//   * a Schur/substitution update  a <- a - l*u  is one fused multiply-add (one rounding),
//     i.e. std::fma(-l, u, a);
//   * a scaling by a pivot p multiplies by the correctly rounded reciprocal r = 1/p;
//   * nothing else is fused (the file is compiled with -ffp-contract=off).
//
// Sources (web pages):
//   [TDLS]  TDLS API, "solver_static.hpp File Reference" (CooperativeLUppSolverStatic),
//           Detailed Description: factorization, factored format, departures from MAGMA.
//   [GLASS] GLASS API reference, "Block-tridiagonal Ops", sections "Direct solve
//           (glass::bdsv)" and "Block-tridiagonal matrix-vector product".
//   [RUDA]  RUDA docs, "ruSOLVER: small-matrix kernel optimisation", section on the
//           unchanged numerical and failure contract.
//   [cuSolverDx] cuSolverDx docs, "Cholesky Factorization" (POTRF).
#include <cfloat>
#include <cmath>
#include <utility>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

template <typename T> struct Limits;
template <> struct Limits<float> {
  static float floor_() { return FLT_MIN; }
};
template <> struct Limits<double> {
  static double floor_() { return DBL_MIN; }
};

// Element (r, c) of an n x m matrix stored row-major (layout 0) or column-major (1).
inline int64_t at(int layout, int rows, int cols, int r, int c) {
  return layout == 0 ? (int64_t)r * cols + c : (int64_t)c * rows + r;
}

// ---------------------------------------------------------------------------------
// LU with partial pivoting, right-looking, in LAPACK's unblocked order ([TDLS]:
// "the right-looking LU with partial pivoting of MAGMA's register-blocked small-system
// kernel ... same operations, same order and, with relative_pivot_threshold = 1, same
// pivot choice"), applied to A itself (P A = L U) whatever the storage order.
//
// Step k:
//   1. pivot search over rows k..n-1 of column k: the first row of largest magnitude
//      in the current row order (lowest-row tie rule, [RUDA]);
//   2. ipiv[k] = p + 1 (1-based LAPACK swap sequence);
//   3. a pivot with !(|pivot| >= smallest normal) is singular ([TDLS] singular_floor
//      default); the first such step sets info = k + 1 and the sweep goes on with a
//      pivot reciprocal of 1 ([TDLS]: "a pivot reciprocal of 1 keeps it finite");
//   4. rows k and p are interchanged in A (whole rows, L part included) and in B;
//   5. multipliers l_ik = a_ik * (1/a_kk) for i > k, stored in place of a_ik;
//   6. rank-1 Schur update a_ij -= l_ik a_kj (i, j > k), and the forward solve
//      b_i -= l_ik b_k folded into the same step ([TDLS]: "L y = P b folded into the
//      factorization").
// Then U x = y by back substitution, column by column from the last:
//   x_k = y_k * (1/u_kk);  y_i -= u_ik x_k for i < k.
// A system with info != 0 returns X = 0 ([RUDA] failed outputs zeroed); its factor
// holds whatever the sweep produced.
//
// tie_step (optional) receives the first step whose two largest candidates lie within
// 1e-6 relative of each other (a near tie, where a different rounding may legitimately
// pick the other row), or -1.
// ---------------------------------------------------------------------------------
// ---------------------------------------------------------------------------------
// Contract variants (the option sets of the _ex calls).
//
// [TDLS] threshold pivoting, Config.relative_pivot_threshold = tau in (0, 1]: "1 keeps
// the choice of MAGMA and LAPACK, a smaller value keeps the row in place more often".
// Reading: with m the magnitude the partial-pivoting search of step k finds (its first
// maximum, the NaN rules of getrf_getrs_one), the row in place stays the pivot when
// |a_kk| >= tau * m, the product rounded in T; otherwise the first maximum is taken.
// tau = 1 is getrf_getrs_one exactly.
//
// [RUDA] status contract ("unchanged numerical and failure contract"): 0 success; k > 0
// the first failing pivot (Cholesky: leading minor); -1 a non-finite input (A or B);
// -2 (Cholesky) an input matrix that is not symmetric; -3 a non-finite intermediate
// result (read here: an entry of the factor or of X that is not finite at the end of a
// sweep that met no failing pivot). A failed system returns its factor and X as zeros
// and, for LU, every pivot entry as -1. Checks run in the order -1, -2, the sweep, -3.
// ---------------------------------------------------------------------------------
template <typename T>
bool all_finite(const T* p, int64_t count) {
  for (int64_t i = 0; i < count; ++i)
    if (!std::isfinite(p[i])) return false;
  return true;
}

template <typename T>
void getrf_getrs_ex_one(int layout, int n, int nrhs, T* A, T* B, int32_t* ipiv, int32_t* info,
                        int32_t* tie_step, T tau, int ruda, int scale = 0) {
  const T floor_v = Limits<T>::floor_();
  auto fail_ruda = [&](int32_t code) {
    for (int i = 0; i < n * n; ++i) A[i] = T(0);
    for (int i = 0; i < n * nrhs; ++i) B[i] = T(0);
    for (int k = 0; k < n; ++k) ipiv[k] = -1;
    *info = code;
  };
  if (ruda && !(all_finite(A, (int64_t)n * n) && all_finite(B, (int64_t)n * nrhs))) {
    fail_ruda(-1);
    if (tie_step) *tie_step = -1;
    return;
  }
  // [RUDA] scaling by the largest magnitude of the whole matrix: when it is finite and
  // positive, every entry is divided by it before the sweep and U gets the scale back
  // after it (U <- U * m, the diagonal included; L is scale-free)
  T msc = T(0);
  if (scale && all_finite(A, (int64_t)n * n)) {
    for (int i = 0; i < n * n; ++i)
      if (std::fabs(A[i]) > msc) msc = std::fabs(A[i]);
    if (msc > T(0))
      for (int i = 0; i < n * n; ++i) A[i] = A[i] / msc;
  }
  int32_t inf = 0;
  int32_t tie = -1;
  auto a = [&](int r, int c) -> T& { return A[at(layout, n, n, r, c)]; };
  auto b = [&](int r, int c) -> T& { return B[at(layout, n, nrhs, r, c)]; };
  for (int k = 0; k < n; ++k) {
    int p = k;
    T best = std::fabs(a(k, k));
    for (int i = k + 1; i < n; ++i) {
      T v = std::fabs(a(i, k));
      if (v > best) {
        best = v;
        p = i;
      }
    }
    if (tie < 0 && best > T(0)) {
      T second = T(-1);
      for (int i = k; i < n; ++i) {
        if (i == p) continue;
        T v = std::fabs(a(i, k));
        if (v > second) second = v;
      }
      if (second >= T(0) && (double)best - (double)second <= 1e-6 * (double)best) tie = k;
    }
    const T akk = std::fabs(a(k, k));
    if (p != k && tau < T(1)) {
      const T bar = tau * best;
      if (tie < 0 && std::fabs((double)akk - (double)bar) <= 1e-6 * (double)best) tie = k;
      if (akk >= bar) p = k;   // the row in place is kept
    }
    const T mag = (p == k) ? akk : best;
    ipiv[k] = p + 1;
    const bool ok = mag >= floor_v;
    if (!ok && inf == 0) inf = k + 1;
    if (p != k) {
      for (int c = 0; c < n; ++c) {
        T t = a(k, c);
        a(k, c) = a(p, c);
        a(p, c) = t;
      }
      for (int c = 0; c < nrhs; ++c) {
        T t = b(k, c);
        b(k, c) = b(p, c);
        b(p, c) = t;
      }
    }
    const T r = ok ? T(1) / a(k, k) : T(1);
    for (int i = k + 1; i < n; ++i) a(i, k) = a(i, k) * r;
    for (int i = k + 1; i < n; ++i) {
      const T l = a(i, k);
      for (int j = k + 1; j < n; ++j) a(i, j) = std::fma(-l, a(k, j), a(i, j));
      for (int c = 0; c < nrhs; ++c) b(i, c) = std::fma(-l, b(k, c), b(i, c));
    }
  }
  if (msc > T(0))
    for (int k = 0; k < n; ++k)
      for (int j = k; j < n; ++j) a(k, j) = a(k, j) * msc;   // U's scale restored
  for (int k = n - 1; k >= 0; --k) {
    const T piv = a(k, k);
    const T r = (std::fabs(piv) >= floor_v) ? T(1) / piv : T(1);
    for (int c = 0; c < nrhs; ++c) {
      const T x = b(k, c) * r;
      b(k, c) = x;
      for (int i = 0; i < k; ++i) b(i, c) = std::fma(-a(i, k), x, b(i, c));
    }
  }
  if (tie_step) *tie_step = tie;
  if (ruda && inf == 0 && !(all_finite(A, (int64_t)n * n) && all_finite(B, (int64_t)n * nrhs)))
    inf = -3;
  if (inf != 0) {
    if (ruda) {
      fail_ruda(inf);
      return;
    }
    for (int i = 0; i < n * nrhs; ++i) B[i] = T(0);
  }
  *info = inf;
}

template <typename T>
void getrf_getrs_one(int layout, int n, int nrhs, T* A, T* B, int32_t* ipiv, int32_t* info,
                     int32_t* tie_step) {
  // partial pivoting (tau = 1) under the default contract: the steps listed above
  getrf_getrs_ex_one<T>(layout, n, nrhs, A, B, ipiv, info, tie_step, T(1), 0);
}

// ---------------------------------------------------------------------------------
// getrs: solve with a stored factor ([TDLS] separate substitution; [GLASS] "factor once,
// call this per right-hand side"). LU holds L\U as left by getrf_getrs_one (nrhs = 0 gives
// getrf), ipiv the 1-based swap sequence. B <- X:
//   1. the interchanges in step order: rows k and ipiv[k]-1 of B for k = 0..n-1 (an
//      entry outside 1..n swaps nothing: the solve steps take no status to report it);
//   2. L y = P b with unit L, column by column: b_i -= l_ik b_k for i > k (each b_i takes
//      its updates in increasing k, as in the fused sweep);
//   3. U x = y as in getrf_getrs_one, a pivot reciprocal of 1 for a singular u_kk.
// No info: a factor whose info != 0 gives an unspecified (finite or not) X.
// ---------------------------------------------------------------------------------
template <typename T>
void getrs_one(int layout, int n, int nrhs, const T* LU, const int32_t* ipiv, T* B) {
  const T floor_v = Limits<T>::floor_();
  auto a = [&](int r, int c) -> T { return LU[at(layout, n, n, r, c)]; };
  auto b = [&](int r, int c) -> T& { return B[at(layout, n, nrhs, r, c)]; };
  for (int k = 0; k < n; ++k) {
    const int p = ipiv[k] - 1;
    if (p != k && p >= 0 && p < n)
      for (int c = 0; c < nrhs; ++c) {
        T t = b(k, c);
        b(k, c) = b(p, c);
        b(p, c) = t;
      }
  }
  for (int k = 0; k < n; ++k)
    for (int i = k + 1; i < n; ++i) {
      const T l = a(i, k);
      for (int c = 0; c < nrhs; ++c) b(i, c) = std::fma(-l, b(k, c), b(i, c));
    }
  for (int k = n - 1; k >= 0; --k) {
    const T piv = a(k, k);
    const T r = (std::fabs(piv) >= floor_v) ? T(1) / piv : T(1);
    for (int c = 0; c < nrhs; ++c) {
      const T x = b(k, c) * r;
      b(k, c) = x;
      for (int i = 0; i < k; ++i) b(i, c) = std::fma(-a(i, k), x, b(i, c));
    }
  }
}

// ---------------------------------------------------------------------------------
// Cholesky, lower fill, right-looking ([cuSolverDx] POTRF: only the lower triangle is
// read and replaced by L, the upper part is untouched; info = the smallest leading
// minor that is not positive definite). Column k:
//   d = a_kk (already updated); !(d > 0) -> info = k + 1 and the remaining columns
//   are left as they are; l_kk = sqrt(d); l_ik = a_ik * (1/l_kk) for i > k;
//   a_ij -= l_ik l_jk for k < j <= i.
// potrs: L y = b (column by column, y_k = b_k * (1/l_kk), b_i -= l_ik y_k for i > k),
// then L^T x = y (from the last: x_k = y_k * (1/l_kk), y_i -= l_ki x_k for i < k).
// A failed system returns X = 0.
// Upper fill ([cuSolverDx]: A = U^T U, only the upper triangle processed and replaced by
// U, the lower part untouched): U is L^T for the lower factor of the mirrored matrix, and
// the upper algorithm's operations are the lower algorithm's on mirrored entries. A in
// layout X with upper fill is therefore read as the lower fill of A in the other layout
// (a_layout = 1 - X), while B keeps its own layout.
// ---------------------------------------------------------------------------------
template <typename T>
void potrf_potrs_one(int a_layout, int b_layout, int n, int nrhs, T* A, T* B, int32_t* info) {
  int32_t inf = 0;
  auto a = [&](int r, int c) -> T& { return A[at(a_layout, n, n, r, c)]; };
  auto b = [&](int r, int c) -> T& { return B[at(b_layout, n, nrhs, r, c)]; };
  for (int k = 0; k < n; ++k) {
    const T d = a(k, k);
    if (!(d > T(0))) {
      inf = k + 1;
      break;
    }
    const T l = std::sqrt(d);
    a(k, k) = l;
    const T r = T(1) / l;
    for (int i = k + 1; i < n; ++i) a(i, k) = a(i, k) * r;
    for (int j = k + 1; j < n; ++j) {
      const T ljk = a(j, k);
      for (int i = j; i < n; ++i) a(i, j) = std::fma(-a(i, k), ljk, a(i, j));
    }
  }
  if (inf != 0) {
    for (int r0 = 0; r0 < n; ++r0)
      for (int c = 0; c < nrhs; ++c) b(r0, c) = T(0);
    *info = inf;
    return;
  }
  for (int c = 0; c < nrhs; ++c) {
    for (int k = 0; k < n; ++k) {
      const T y = b(k, c) * (T(1) / a(k, k));
      b(k, c) = y;
      for (int i = k + 1; i < n; ++i) b(i, c) = std::fma(-a(i, k), y, b(i, c));
    }
    for (int k = n - 1; k >= 0; --k) {
      const T x = b(k, c) * (T(1) / a(k, k));
      b(k, c) = x;
      for (int i = 0; i < k; ++i) b(i, c) = std::fma(-a(k, i), x, b(i, c));
    }
  }
  *info = 0;
}

// potrs with a stored lower factor L (potrf_potrs_one with nrhs = 0 gives potrf): the
// solve half of potrf_potrs_one, with the same operation order. No info: a failed factor
// gives an unspecified X.
template <typename T>
void potrs_one(int a_layout, int b_layout, int n, int nrhs, const T* L, T* B) {
  auto a = [&](int r, int c) -> T { return L[at(a_layout, n, n, r, c)]; };
  auto b = [&](int r, int c) -> T& { return B[at(b_layout, n, nrhs, r, c)]; };
  for (int c = 0; c < nrhs; ++c) {
    for (int k = 0; k < n; ++k) {
      const T y = b(k, c) * (T(1) / a(k, k));
      b(k, c) = y;
      for (int i = k + 1; i < n; ++i) b(i, c) = std::fma(-a(i, k), y, b(i, c));
    }
    for (int k = n - 1; k >= 0; --k) {
      const T x = b(k, c) * (T(1) / a(k, k));
      b(k, c) = x;
      for (int i = 0; i < k; ++i) b(i, c) = std::fma(-a(k, i), x, b(i, c));
    }
  }
}

// ---------------------------------------------------------------------------------
// Block-tridiagonal SPD solve by the block-Cholesky (block-Thomas) sweep ([GLASS]
// bdsv_factor / bdsv_solve / bdsv).
// Layout ([GLASS]): block-row br is a bs x (3 bs) row-major strip [L | D | R] at
// strips + br*3*bs*bs; slot (y, x) of sub-block s lives at strip[y*3bs + s*bs + x].
// The vector is padded: (nbr + 2)*bs entries, block-row br at (br + 1)*bs.
// Factor: F_0 = chol(D_0); for k > 0: E_k = L_k F_{k-1}^{-T}, F_k = chol(D_k - E_k E_k^T).
//   MAIN <- F_k (lower triangle; the upper triangle keeps D_k), LEFT <- E_k, RIGHT is
//   neither read nor written.
// Solve: y_k = F_k^{-1}(b_k - E_k y_{k-1}), then x_k = F_k^{-T}(y_k - E_{k+1}^T x_{k+1}).
// info = global index br*bs + j + 1 of the first failing diagonal of the sweep (the
// dense Cholesky factor of the assembled matrix fails at the same index). GLASS only
// raises a flag and runs the sweep on; this oracle stops at the first failure, the
// strips beyond it are then unspecified and the solution is returned as zeros.
// ---------------------------------------------------------------------------------
// Offset of slot (y, x) of sub-block `slot` (0 = LEFT, 1 = MAIN, 2 = RIGHT) of block-row br.
inline int64_t strip_at(int bs, int br, int slot, int y, int x) {
  const int w = 3 * bs;
  return (int64_t)br * bs * w + (int64_t)y * w + slot * bs + x;
}

// bdsv_factor: the factor sweep, in place on the strips; returns info (0 or the global
// index of the first failing diagonal, where the sweep stops).
template <typename T>
int32_t bdsv_factor_one(int nbr, int bs, T* strips) {
  auto blk = [&](int br, int slot, int y, int x) -> T& {
    return strips[strip_at(bs, br, slot, y, x)];
  };
  const int LEFT = 0, MAIN = 1;
  int32_t inf = 0;
  std::vector<T> S((size_t)bs * bs), E((size_t)bs * bs);
  for (int k = 0; k < nbr && inf == 0; ++k) {
    // S = D_k (lower triangle), minus E_k E_k^T for k > 0.
    for (int i = 0; i < bs; ++i)
      for (int j = 0; j <= i; ++j) S[i * bs + j] = blk(k, MAIN, i, j);
    if (k > 0) {
      // E_k = L_k F_{k-1}^{-T}: row a solves e_a F^T = l_a, i.e. for j = 0..bs-1
      // e_aj = (l_aj - sum_{m<j} e_am f_jm) * (1/f_jj).
      for (int ar = 0; ar < bs; ++ar) {
        for (int j = 0; j < bs; ++j) {
          T s = blk(k, LEFT, ar, j);
          for (int m = 0; m < j; ++m) s = std::fma(-E[ar * bs + m], blk(k - 1, MAIN, j, m), s);
          E[ar * bs + j] = s * (T(1) / blk(k - 1, MAIN, j, j));
        }
      }
      for (int i = 0; i < bs; ++i)
        for (int j = 0; j <= i; ++j) {
          T s = S[i * bs + j];
          for (int m = 0; m < bs; ++m) s = std::fma(-E[i * bs + m], E[j * bs + m], s);
          S[i * bs + j] = s;
        }
      for (int i = 0; i < bs; ++i)
        for (int j = 0; j < bs; ++j) blk(k, LEFT, i, j) = E[i * bs + j];
    }
    // F_k = chol(S), right-looking as in potrf_potrs_one.
    for (int c = 0; c < bs; ++c) {
      const T d = S[c * bs + c];
      if (!(d > T(0))) {
        inf = k * bs + c + 1;
        break;
      }
      const T l = std::sqrt(d);
      S[c * bs + c] = l;
      const T r = T(1) / l;
      for (int i = c + 1; i < bs; ++i) S[i * bs + c] = S[i * bs + c] * r;
      for (int j = c + 1; j < bs; ++j) {
        const T ljc = S[j * bs + c];
        for (int i = j; i < bs; ++i) S[i * bs + j] = std::fma(-S[i * bs + c], ljc, S[i * bs + j]);
      }
    }
    for (int i = 0; i < bs; ++i)
      for (int j = 0; j <= i; ++j) blk(k, MAIN, i, j) = S[i * bs + j];
  }
  return inf;
}

// bdsv_solve: forward then backward block substitution on the interior of the padded
// vector, with strips factored by bdsv_factor_one (read only).
template <typename T>
void bdsv_solve_one(int nbr, int bs, const T* strips, T* xpad) {
  auto blk = [&](int br, int slot, int y, int x) -> T { return strips[strip_at(bs, br, slot, y, x)]; };
  const int LEFT = 0, MAIN = 1;
  T* x = xpad + bs;  // interior: block-row br at x + br*bs
  std::vector<T> z(bs);
  // Forward sweep: z = b_k - E_k y_{k-1}; y_k = F_k^{-1} z.
  for (int k = 0; k < nbr; ++k) {
    for (int i = 0; i < bs; ++i) z[i] = x[k * bs + i];
    if (k > 0)
      for (int i = 0; i < bs; ++i)
        for (int m = 0; m < bs; ++m) z[i] = std::fma(-blk(k, LEFT, i, m), x[(k - 1) * bs + m], z[i]);
    for (int j = 0; j < bs; ++j) {
      T s = z[j];
      for (int m = 0; m < j; ++m) s = std::fma(-blk(k, MAIN, j, m), x[k * bs + m], s);
      x[k * bs + j] = s * (T(1) / blk(k, MAIN, j, j));
    }
  }
  // Backward sweep: w = y_k - E_{k+1}^T x_{k+1}; x_k = F_k^{-T} w.
  for (int k = nbr - 1; k >= 0; --k) {
    for (int i = 0; i < bs; ++i) z[i] = x[k * bs + i];
    if (k < nbr - 1)
      for (int m = 0; m < bs; ++m)
        for (int i = 0; i < bs; ++i) z[m] = std::fma(-blk(k + 1, LEFT, i, m), x[(k + 1) * bs + i], z[m]);
    for (int j = bs - 1; j >= 0; --j) {
      T s = z[j];
      for (int m = j + 1; m < bs; ++m) s = std::fma(-blk(k, MAIN, m, j), x[k * bs + m], s);
      x[k * bs + j] = s * (T(1) / blk(k, MAIN, j, j));
    }
  }
}

// bdsv = bdsv_factor then bdsv_solve; a failed factor returns the interior as zeros.
template <typename T>
void bdsv_one(int nbr, int bs, T* strips, T* xpad, int32_t* info) {
  const int32_t inf = bdsv_factor_one(nbr, bs, strips);
  if (inf != 0) {
    for (int i = 0; i < nbr * bs; ++i) xpad[bs + i] = T(0);
    *info = inf;
    return;
  }
  bdsv_solve_one(nbr, bs, strips, xpad);
  *info = 0;
}

// ---------------------------------------------------------------------------------
// bdmv ([GLASS] "Block-tridiagonal matrix-vector product"): y = A x with A given by the
// strips [L | D | R] (all three blocks as stored) and padded vectors. Block-row br reads
// the window x[br*bs, br*bs + 3bs) (previous / current / next block) and writes
// y[(br+1)*bs + row]; the pad blocks of y are left as they are. The pages fix no
// summation order (only that the result does not depend on the thread count): here each
// entry is one dot product over its strip row in increasing column order, one fused
// multiply-add per term, starting from zero.
// ---------------------------------------------------------------------------------
template <typename T>
void bdmv_one(int nbr, int bs, const T* strips, const T* xpad, T* ypad) {
  const int w = 3 * bs;
  for (int br = 0; br < nbr; ++br)
    for (int row = 0; row < bs; ++row) {
      const T* srow = strips + strip_at(bs, br, 0, row, 0);
      const T* xw = xpad + (int64_t)br * bs;
      T acc = T(0);
      for (int c = 0; c < w; ++c) acc = std::fma(srow[c], xw[c], acc);
      ypad[(int64_t)(br + 1) * bs + row] = acc;
    }
}

// [TDLS] the row-major reading: the solver factors S, the stored matrix read column-major
// (S = A^T for row-major storage): P S = L U, so A = U^T L^T P, and the solve is the
// mirror of the default one: U^T z = b (column by column: z_k = b_k * r_k, then
// b_j -= u_kj z_k for j > k, in increasing k; r_k as in getrs), L^T w = z (unit
// diagonal, from the last: b_i -= l_ki w_k for i < k, in decreasing k), x = P^T w (the
// swaps applied to w in reverse step order). The factor is getrf_getrs_ex_one's on the
// memory read column-major; B keeps its storage order. Under column-major storage S = A
// and TDLS's solve is the default one.
template <typename T>
void getrs_mirror_one(int b_layout, int n, int nrhs, const T* S, const int32_t* ipiv, T* B) {
  const T floor_v = Limits<T>::floor_();
  auto s_ = [&](int r, int c) -> T { return S[at(1, n, n, r, c)]; };
  auto b = [&](int r, int c) -> T& { return B[at(b_layout, n, nrhs, r, c)]; };
  for (int k = 0; k < n; ++k) {
    const T piv = s_(k, k);
    const T r = (std::fabs(piv) >= floor_v) ? T(1) / piv : T(1);
    for (int c = 0; c < nrhs; ++c) {
      const T z = b(k, c) * r;
      b(k, c) = z;
      for (int j = k + 1; j < n; ++j) b(j, c) = std::fma(-s_(k, j), z, b(j, c));
    }
  }
  for (int k = n - 1; k >= 0; --k)
    for (int c = 0; c < nrhs; ++c)
      for (int i = 0; i < k; ++i) b(i, c) = std::fma(-s_(k, i), b(k, c), b(i, c));
  for (int k = n - 1; k >= 0; --k) {  // x = P^T w: step k's interchange undone
    const int q = ipiv[k] - 1;
    if (q == k || q < 0 || q >= n) continue;   // out of range: no interchange
    for (int c = 0; c < nrhs; ++c) std::swap(b(k, c), b(q, c));
  }
}

template <typename T>
void potrf_potrs_ex_one(int a_layout, int b_layout, int n, int nrhs, T* A, T* B, int32_t* info,
                        int ruda) {
  auto a = [&](int r, int c) -> T& { return A[at(a_layout, n, n, r, c)]; };
  auto fail_ruda = [&](int32_t code) {
    for (int r = 0; r < n; ++r)
      for (int c = 0; c <= r; ++c) a(r, c) = T(0);   // the factor's triangle
    for (int i = 0; i < n * nrhs; ++i) B[i] = T(0);
    *info = code;
  };
  if (ruda) {
    if (!(all_finite(A, (int64_t)n * n) && all_finite(B, (int64_t)n * nrhs))) {
      fail_ruda(-1);
      return;
    }
    for (int r = 0; r < n; ++r)
      for (int c = 0; c < r; ++c)
        if (!(a(r, c) == a(c, r))) {
          fail_ruda(-2);
          return;
        }
  }
  potrf_potrs_one<T>(a_layout, b_layout, n, nrhs, A, B, info);
  if (!ruda) return;
  int32_t inf = *info;
  if (inf == 0) {
    bool fin = all_finite(B, (int64_t)n * nrhs);
    for (int r = 0; r < n && fin; ++r)
      for (int c = 0; c <= r; ++c)
        if (!std::isfinite(a(r, c))) {
          fin = false;
          break;
        }
    if (!fin) inf = -3;
  }
  if (inf != 0) fail_ruda(inf);
}

// Hands contiguous ranges of systems to nthreads workers (1 = the calling thread).
template <typename F>
void for_systems(int64_t batch, int nthreads, F&& f) {
  if (nthreads <= 1 || batch < 2) {
    for (int64_t s = 0; s < batch; ++s) f(s);
    return;
  }
  if ((int64_t)nthreads > batch) nthreads = (int)batch;
  std::vector<std::thread> pool;
  pool.reserve(nthreads);
  for (int t = 0; t < nthreads; ++t) {
    const int64_t lo = batch * t / nthreads, hi = batch * (t + 1) / nthreads;
    pool.emplace_back([lo, hi, &f] {
      for (int64_t s = lo; s < hi; ++s) f(s);
    });
  }
  for (auto& th : pool) th.join();
}

template <typename T>
int getrf_getrs_batched(int layout, int n, int nrhs, int64_t batch, T* A, T* B, int32_t* ipiv,
                        int32_t* info, int32_t* tie_step, int nthreads) {
  if ((layout != 0 && layout != 1) || n < 1 || nrhs < 1 || batch < 0) return 1;
  for_systems(batch, nthreads, [&](int64_t s) {
    getrf_getrs_one<T>(layout, n, nrhs, A + s * n * n, B + s * n * nrhs, ipiv + s * n, info + s,
                       tie_step ? tie_step + s : nullptr);
  });
  return 0;
}

template <typename T>
int potrf_potrs_batched(int layout, int fill, int n, int nrhs, int64_t batch, T* A, T* B,
                        int32_t* info, int nthreads) {
  if ((layout != 0 && layout != 1) || (fill != 0 && fill != 1) || n < 1 || nrhs < 1 || batch < 0)
    return 1;
  const int a_layout = fill == 0 ? layout : 1 - layout;
  for_systems(batch, nthreads, [&](int64_t s) {
    potrf_potrs_one<T>(a_layout, layout, n, nrhs, A + s * n * n, B + s * n * nrhs, info + s);
  });
  return 0;
}

template <typename T>
int bdsv_batched(int nbr, int bs, int64_t batch, T* strips, T* xpad, int32_t* info, int nthreads) {
  if (nbr < 1 || bs < 1 || batch < 0) return 1;
  const int64_t sstride = (int64_t)nbr * bs * 3 * bs, vstride = (int64_t)(nbr + 2) * bs;
  for_systems(batch, nthreads, [&](int64_t s) {
    bdsv_one<T>(nbr, bs, strips + s * sstride, xpad + s * vstride, info + s);
  });
  return 0;
}

template <typename T>
int getrf_batched(int layout, int n, int64_t batch, T* A, int32_t* ipiv, int32_t* info,
                  int32_t* tie_step, int nthreads) {
  if ((layout != 0 && layout != 1) || n < 1 || batch < 0) return 1;
  for_systems(batch, nthreads, [&](int64_t s) {
    getrf_getrs_one<T>(layout, n, 0, A + s * n * n, nullptr, ipiv + s * n, info + s,
                       tie_step ? tie_step + s : nullptr);
  });
  return 0;
}

template <typename T>
int getrs_batched(int layout, int n, int nrhs, int64_t batch, const T* LU, const int32_t* ipiv,
                  T* B, int nthreads) {
  if ((layout != 0 && layout != 1) || n < 1 || nrhs < 1 || batch < 0) return 1;
  for_systems(batch, nthreads, [&](int64_t s) {
    getrs_one<T>(layout, n, nrhs, LU + s * n * n, ipiv + s * n, B + s * n * nrhs);
  });
  return 0;
}

template <typename T>
int potrf_batched(int layout, int fill, int n, int64_t batch, T* A, int32_t* info, int nthreads) {
  if ((layout != 0 && layout != 1) || (fill != 0 && fill != 1) || n < 1 || batch < 0) return 1;
  const int a_layout = fill == 0 ? layout : 1 - layout;
  for_systems(batch, nthreads, [&](int64_t s) {
    potrf_potrs_one<T>(a_layout, layout, n, 0, A + s * n * n, nullptr, info + s);
  });
  return 0;
}

template <typename T>
int potrs_batched(int layout, int fill, int n, int nrhs, int64_t batch, const T* L, T* B,
                  int nthreads) {
  if ((layout != 0 && layout != 1) || (fill != 0 && fill != 1) || n < 1 || nrhs < 1 || batch < 0)
    return 1;
  const int a_layout = fill == 0 ? layout : 1 - layout;
  for_systems(batch, nthreads, [&](int64_t s) {
    potrs_one<T>(a_layout, layout, n, nrhs, L + s * n * n, B + s * n * nrhs);
  });
  return 0;
}

template <typename T>
int bdsv_factor_batched(int nbr, int bs, int64_t batch, T* strips, int32_t* info, int nthreads) {
  if (nbr < 1 || bs < 1 || batch < 0) return 1;
  const int64_t sstride = (int64_t)nbr * bs * 3 * bs;
  for_systems(batch, nthreads, [&](int64_t s) {
    info[s] = bdsv_factor_one<T>(nbr, bs, strips + s * sstride);
  });
  return 0;
}

template <typename T>
int bdsv_solve_batched(int nbr, int bs, int64_t batch, const T* strips, T* xpad, int nthreads) {
  if (nbr < 1 || bs < 1 || batch < 0) return 1;
  const int64_t sstride = (int64_t)nbr * bs * 3 * bs, vstride = (int64_t)(nbr + 2) * bs;
  for_systems(batch, nthreads, [&](int64_t s) {
    bdsv_solve_one<T>(nbr, bs, strips + s * sstride, xpad + s * vstride);
  });
  return 0;
}

template <typename T>
int bdmv_batched(int nbr, int bs, int64_t batch, const T* strips, const T* xpad, T* ypad,
                 int nthreads) {
  if (nbr < 1 || bs < 1 || batch < 0) return 1;
  const int64_t sstride = (int64_t)nbr * bs * 3 * bs, vstride = (int64_t)(nbr + 2) * bs;
  for_systems(batch, nthreads, [&](int64_t s) {
    bdmv_one<T>(nbr, bs, strips + s * sstride, xpad + s * vstride, ypad + s * vstride);
  });
  return 0;
}

template <typename T>
int getrf_getrs_ex_batched(int layout, int n, int nrhs, int64_t batch, T* A, T* B, int32_t* ipiv,
                           int32_t* info, int32_t* tie_step, double tau, int ruda, int scale,
                           int nthreads) {
  if ((layout != 0 && layout != 1) || n < 1 || nrhs < 1 || batch < 0 || !(tau > 0.0) ||
      !(tau <= 1.0))
    return 1;
  const T t = static_cast<T>(tau);
  for_systems(batch, nthreads, [&](int64_t s) {
    getrf_getrs_ex_one<T>(layout, n, nrhs, A + s * n * n, B + s * n * nrhs, ipiv + s * n,
                          info + s, tie_step ? tie_step + s : nullptr, t, ruda, scale);
  });
  return 0;
}

// [TDLS] row-major reading, one system: factor S (the stored array read column-major,
// S = A^T for row-major storage) in place, then U^T z = b, L^T w = z, x = P^T w; X zeros
// when the factor failed. Column-major storage: S = A and the solve is the default one.
// scale: RUDA's max-abs scaling of the factorization (U restored before the solve).
template <typename T>
void mirror_one(int layout, int n, int nrhs, T* As, T* Bs, int32_t* ipiv, int32_t* inf,
                int32_t* tie, T t, int scale) {
  if (layout == 1) {
    getrf_getrs_ex_one<T>(1, n, nrhs, As, Bs, ipiv, inf, tie, t, 0, scale);
    return;
  }
  getrf_getrs_ex_one<T>(1, n, 0, As, nullptr, ipiv, inf, tie, t, 0, scale);
  getrs_mirror_one<T>(layout, n, nrhs, As, ipiv, Bs);
  if (*inf != 0)
    for (int i = 0; i < n * nrhs; ++i) Bs[i] = T(0);
}

template <typename T>
int potrf_potrs_ex_batched(int layout, int fill, int n, int nrhs, int64_t batch, T* A, T* B,
                           int32_t* info, int ruda, int nthreads) {
  if ((layout != 0 && layout != 1) || (fill != 0 && fill != 1) || n < 1 || nrhs < 1 || batch < 0)
    return 1;
  const int a_layout = fill == 0 ? layout : 1 - layout;
  for_systems(batch, nthreads, [&](int64_t s) {
    potrf_potrs_ex_one<T>(a_layout, layout, n, nrhs, A + s * n * n, B + s * n * nrhs, info + s,
                          ruda);
  });
  return 0;
}

}  // namespace

// [TDLS] batched layouts: element e of system s (e the offset of the element in the
// system's own storage order) lives at base_s[e * stride]; AoS is stride 1 (base_s =
// s * size), SoA stride = the batch, AoSoA stride W with the systems in blocks of W:
// base_s = (s / W) * W * size + s % W. One routine covers all three: it gathers each
// system into a contiguous copy, runs the per-system routine and scatters it back. A, B
// and ipiv are interleaved; info holds one entry per system. The contract options (the
// relative pivot threshold, the RUDA status contract) are the per-system routines' own.
template <typename T>
struct Strided {
  T* p;
  int64_t w;
  int64_t size;   // elements of one system
  T* base(int64_t s) const { return p + (s / w) * w * size + s % w; }
  void gather(int64_t s, T* dst) const {
    const T* b = base(s);
    for (int64_t e = 0; e < size; ++e) dst[e] = b[e * w];
  }
  void scatter(int64_t s, const T* src) const {
    T* b = base(s);
    for (int64_t e = 0; e < size; ++e) b[e * w] = src[e];
  }
};

template <typename T>
int getrf_getrs_mirror_batched(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                               int32_t* ipiv, int32_t* info, int32_t* tie_step, double tau,
                               int nthreads, int64_t w, int scale) {
  if ((layout != 0 && layout != 1) || n < 1 || nrhs < 1 || batch < 0 || !(tau > 0.0) ||
      !(tau <= 1.0) || w < 1)
    return 1;
  const T t = static_cast<T>(tau);
  if (w == 1) {
    for_systems(batch, nthreads, [&](int64_t s) {
      mirror_one<T>(layout, n, nrhs, A + s * n * n, B + s * n * nrhs, ipiv + s * n, info + s,
                    tie_step ? tie_step + s : nullptr, t, scale);
    });
    return 0;
  }
  // [TDLS] interleaved batched layout: each system gathered, solved and scattered back
  const Strided<T> a{A, w, (int64_t)n * n}, b{B, w, (int64_t)n * nrhs};
  const Strided<int32_t> pv{ipiv, w, n};
  for_systems(batch, nthreads, [&](int64_t s) {
    std::vector<T> as(a.size), bs(b.size);
    std::vector<int32_t> ps(n);
    a.gather(s, as.data());
    b.gather(s, bs.data());
    mirror_one<T>(layout, n, nrhs, as.data(), bs.data(), ps.data(), info + s,
                  tie_step ? tie_step + s : nullptr, t, scale);
    a.scatter(s, as.data());
    b.scatter(s, bs.data());
    pv.scatter(s, ps.data());
  });
  return 0;
}

// [TDLS] the separate factor and substitution steps on the interleaved batched layouts:
// the per-system getrf / getrs / potrf / potrs between a gather and a scatter.
template <typename T>
int getrf_il_batched(int layout, int n, int64_t batch, int64_t w, T* A, int32_t* ipiv,
                     int32_t* info, int32_t* tie_step, int nthreads) {
  if ((layout != 0 && layout != 1) || n < 1 || batch < 0 || w < 1) return 1;
  const Strided<T> a{A, w, (int64_t)n * n};
  const Strided<int32_t> pv{ipiv, w, n};
  for_systems(batch, nthreads, [&](int64_t s) {
    std::vector<T> as(a.size);
    std::vector<int32_t> ps(n);
    a.gather(s, as.data());
    getrf_getrs_one<T>(layout, n, 0, as.data(), nullptr, ps.data(), info + s,
                       tie_step ? tie_step + s : nullptr);
    a.scatter(s, as.data());
    pv.scatter(s, ps.data());
  });
  return 0;
}

template <typename T>
int getrs_il_batched(int layout, int n, int nrhs, int64_t batch, int64_t w, const T* LU,
                     const int32_t* ipiv, T* B, int nthreads) {
  if ((layout != 0 && layout != 1) || n < 1 || nrhs < 1 || batch < 0 || w < 1) return 1;
  const Strided<T> a{const_cast<T*>(LU), w, (int64_t)n * n}, b{B, w, (int64_t)n * nrhs};
  const Strided<int32_t> pv{const_cast<int32_t*>(ipiv), w, n};
  for_systems(batch, nthreads, [&](int64_t s) {
    std::vector<T> as(a.size), bs(b.size);
    std::vector<int32_t> ps(n);
    a.gather(s, as.data());
    pv.gather(s, ps.data());
    b.gather(s, bs.data());
    getrs_one<T>(layout, n, nrhs, as.data(), ps.data(), bs.data());
    b.scatter(s, bs.data());
  });
  return 0;
}

template <typename T>
int potrf_il_batched(int layout, int fill, int n, int64_t batch, int64_t w, T* A,
                     int32_t* info, int nthreads) {
  if ((layout != 0 && layout != 1) || (fill != 0 && fill != 1) || n < 1 || batch < 0 || w < 1)
    return 1;
  const int a_layout = fill == 0 ? layout : 1 - layout;
  const Strided<T> a{A, w, (int64_t)n * n};
  for_systems(batch, nthreads, [&](int64_t s) {
    std::vector<T> as(a.size);
    a.gather(s, as.data());
    potrf_potrs_one<T>(a_layout, layout, n, 0, as.data(), nullptr, info + s);
    a.scatter(s, as.data());
  });
  return 0;
}

template <typename T>
int potrs_il_batched(int layout, int fill, int n, int nrhs, int64_t batch, int64_t w,
                     const T* L, T* B, int nthreads) {
  if ((layout != 0 && layout != 1) || (fill != 0 && fill != 1) || n < 1 || nrhs < 1 ||
      batch < 0 || w < 1)
    return 1;
  const int a_layout = fill == 0 ? layout : 1 - layout;
  const Strided<T> a{const_cast<T*>(L), w, (int64_t)n * n}, b{B, w, (int64_t)n * nrhs};
  for_systems(batch, nthreads, [&](int64_t s) {
    std::vector<T> as(a.size), bs(b.size);
    a.gather(s, as.data());
    b.gather(s, bs.data());
    potrs_one<T>(a_layout, layout, n, nrhs, as.data(), bs.data());
    b.scatter(s, bs.data());
  });
  return 0;
}

template <typename T>
int getrf_getrs_il_batched(int layout, int n, int nrhs, int64_t batch, int64_t w, T* A, T* B,
                           int32_t* ipiv, int32_t* info, int32_t* tie_step, double tau, int ruda,
                           int scale, int nthreads) {
  if ((layout != 0 && layout != 1) || n < 1 || nrhs < 1 || batch < 0 || w < 1 ||
      !(tau > 0.0) || !(tau <= 1.0))
    return 1;
  const T t = static_cast<T>(tau);
  const Strided<T> a{A, w, (int64_t)n * n}, b{B, w, (int64_t)n * nrhs};
  const Strided<int32_t> pv{ipiv, w, n};
  for_systems(batch, nthreads, [&](int64_t s) {
    std::vector<T> as(a.size), bs(b.size);
    std::vector<int32_t> ps(n);
    a.gather(s, as.data());
    b.gather(s, bs.data());
    getrf_getrs_ex_one<T>(layout, n, nrhs, as.data(), bs.data(), ps.data(), info + s,
                          tie_step ? tie_step + s : nullptr, t, ruda, scale);
    a.scatter(s, as.data());
    b.scatter(s, bs.data());
    pv.scatter(s, ps.data());
  });
  return 0;
}

template <typename T>
int potrf_potrs_il_batched(int layout, int fill, int n, int nrhs, int64_t batch, int64_t w, T* A,
                           T* B, int32_t* info, int ruda, int nthreads) {
  if ((layout != 0 && layout != 1) || (fill != 0 && fill != 1) || n < 1 || nrhs < 1 ||
      batch < 0 || w < 1)
    return 1;
  const int a_layout = fill == 0 ? layout : 1 - layout;
  const Strided<T> a{A, w, (int64_t)n * n}, b{B, w, (int64_t)n * nrhs};
  for_systems(batch, nthreads, [&](int64_t s) {
    std::vector<T> as(a.size), bs(b.size);
    a.gather(s, as.data());
    b.gather(s, bs.data());
    potrf_potrs_ex_one<T>(a_layout, layout, n, nrhs, as.data(), bs.data(), info + s, ruda);
    a.scatter(s, as.data());
    b.scatter(s, bs.data());
  });
  return 0;
}

extern "C" {

int oracle_getrf_getrs_f32(int layout, int n, int nrhs, int64_t batch, float* A, float* B,
                           int32_t* ipiv, int32_t* info, int32_t* tie_step, int nthreads) {
  return getrf_getrs_batched<float>(layout, n, nrhs, batch, A, B, ipiv, info, tie_step, nthreads);
}
int oracle_getrf_getrs_f64(int layout, int n, int nrhs, int64_t batch, double* A, double* B,
                           int32_t* ipiv, int32_t* info, int32_t* tie_step, int nthreads) {
  return getrf_getrs_batched<double>(layout, n, nrhs, batch, A, B, ipiv, info, tie_step, nthreads);
}
int oracle_potrf_potrs_f32(int layout, int fill, int n, int nrhs, int64_t batch, float* A, float* B,
                           int32_t* info, int nthreads) {
  return potrf_potrs_batched<float>(layout, fill, n, nrhs, batch, A, B, info, nthreads);
}
int oracle_potrf_potrs_f64(int layout, int fill, int n, int nrhs, int64_t batch, double* A, double* B,
                           int32_t* info, int nthreads) {
  return potrf_potrs_batched<double>(layout, fill, n, nrhs, batch, A, B, info, nthreads);
}
int oracle_bdsv_f32(int nbr, int bs, int64_t batch, float* strips, float* xpad, int32_t* info,
                    int nthreads) {
  return bdsv_batched<float>(nbr, bs, batch, strips, xpad, info, nthreads);
}
int oracle_bdsv_f64(int nbr, int bs, int64_t batch, double* strips, double* xpad, int32_t* info,
                    int nthreads) {
  return bdsv_batched<double>(nbr, bs, batch, strips, xpad, info, nthreads);
}

int oracle_getrf_f32(int layout, int n, int64_t batch, float* A, int32_t* ipiv, int32_t* info,
                     int32_t* tie_step, int nthreads) {
  return getrf_batched<float>(layout, n, batch, A, ipiv, info, tie_step, nthreads);
}
int oracle_getrs_f32(int layout, int n, int nrhs, int64_t batch, const float* LU,
                     const int32_t* ipiv, float* B, int nthreads) {
  return getrs_batched<float>(layout, n, nrhs, batch, LU, ipiv, B, nthreads);
}
int oracle_potrf_f32(int layout, int fill, int n, int64_t batch, float* A, int32_t* info,
                     int nthreads) {
  return potrf_batched<float>(layout, fill, n, batch, A, info, nthreads);
}
int oracle_potrs_f32(int layout, int fill, int n, int nrhs, int64_t batch, const float* L, float* B,
                     int nthreads) {
  return potrs_batched<float>(layout, fill, n, nrhs, batch, L, B, nthreads);
}
int oracle_bdsv_factor_f32(int nbr, int bs, int64_t batch, float* strips, int32_t* info,
                           int nthreads) {
  return bdsv_factor_batched<float>(nbr, bs, batch, strips, info, nthreads);
}
int oracle_bdsv_solve_f32(int nbr, int bs, int64_t batch, const float* strips, float* xpad,
                          int nthreads) {
  return bdsv_solve_batched<float>(nbr, bs, batch, strips, xpad, nthreads);
}
int oracle_bdmv_f32(int nbr, int bs, int64_t batch, const float* strips, const float* xpad,
                    float* ypad, int nthreads) {
  return bdmv_batched<float>(nbr, bs, batch, strips, xpad, ypad, nthreads);
}
int oracle_getrf_f64(int layout, int n, int64_t batch, double* A, int32_t* ipiv, int32_t* info,
                     int32_t* tie_step, int nthreads) {
  return getrf_batched<double>(layout, n, batch, A, ipiv, info, tie_step, nthreads);
}
int oracle_getrs_f64(int layout, int n, int nrhs, int64_t batch, const double* LU,
                     const int32_t* ipiv, double* B, int nthreads) {
  return getrs_batched<double>(layout, n, nrhs, batch, LU, ipiv, B, nthreads);
}
int oracle_potrf_f64(int layout, int fill, int n, int64_t batch, double* A, int32_t* info,
                     int nthreads) {
  return potrf_batched<double>(layout, fill, n, batch, A, info, nthreads);
}
int oracle_potrs_f64(int layout, int fill, int n, int nrhs, int64_t batch, const double* L, double* B,
                     int nthreads) {
  return potrs_batched<double>(layout, fill, n, nrhs, batch, L, B, nthreads);
}
int oracle_bdsv_factor_f64(int nbr, int bs, int64_t batch, double* strips, int32_t* info,
                           int nthreads) {
  return bdsv_factor_batched<double>(nbr, bs, batch, strips, info, nthreads);
}
int oracle_bdsv_solve_f64(int nbr, int bs, int64_t batch, const double* strips, double* xpad,
                          int nthreads) {
  return bdsv_solve_batched<double>(nbr, bs, batch, strips, xpad, nthreads);
}
int oracle_bdmv_f64(int nbr, int bs, int64_t batch, const double* strips, const double* xpad,
                    double* ypad, int nthreads) {
  return bdmv_batched<double>(nbr, bs, batch, strips, xpad, ypad, nthreads);
}
int oracle_getrf_getrs_ex_f32(int layout, int n, int nrhs, int64_t batch, float* A, float* B,
                              int32_t* ipiv, int32_t* info, int32_t* tie_step, double tau,
                              int ruda, int scale, int nthreads) {
  return getrf_getrs_ex_batched<float>(layout, n, nrhs, batch, A, B, ipiv, info, tie_step, tau,
                                     ruda, scale, nthreads);
}
int oracle_potrf_potrs_ex_f32(int layout, int fill, int n, int nrhs, int64_t batch, float* A,
                              float* B, int32_t* info, int ruda, int nthreads) {
  return potrf_potrs_ex_batched<float>(layout, fill, n, nrhs, batch, A, B, info, ruda, nthreads);
}
int oracle_getrf_getrs_ex_f64(int layout, int n, int nrhs, int64_t batch, double* A, double* B,
                              int32_t* ipiv, int32_t* info, int32_t* tie_step, double tau,
                              int ruda, int scale, int nthreads) {
  return getrf_getrs_ex_batched<double>(layout, n, nrhs, batch, A, B, ipiv, info, tie_step, tau,
                                     ruda, scale, nthreads);
}
int oracle_potrf_potrs_ex_f64(int layout, int fill, int n, int nrhs, int64_t batch, double* A,
                              double* B, int32_t* info, int ruda, int nthreads) {
  return potrf_potrs_ex_batched<double>(layout, fill, n, nrhs, batch, A, B, info, ruda, nthreads);
}
int oracle_getrf_getrs_mirror_f32(int layout, int n, int nrhs, int64_t batch, float* A, float* B,
                                  int32_t* ipiv, int32_t* info, int32_t* tie_step, double tau,
                                  int nthreads) {
  return getrf_getrs_mirror_batched<float>(layout, n, nrhs, batch, A, B, ipiv, info, tie_step, tau,
                                         nthreads, 1, 0);
}
int oracle_getrf_getrs_mirror_f64(int layout, int n, int nrhs, int64_t batch, double* A, double* B,
                                  int32_t* ipiv, int32_t* info, int32_t* tie_step, double tau,
                                  int nthreads) {
  return getrf_getrs_mirror_batched<double>(layout, n, nrhs, batch, A, B, ipiv, info, tie_step, tau,
                                         nthreads, 1, 0);
}
int oracle_getrf_getrs_il_f32(int layout, int n, int nrhs, int64_t batch, int64_t w, float* A,
                              float* B, int32_t* ipiv, int32_t* info, int32_t* tie_step,
                              double tau, int ruda, int scale, int nthreads) {
  return getrf_getrs_il_batched<float>(layout, n, nrhs, batch, w, A, B, ipiv, info, tie_step,
                                     tau, ruda, scale, nthreads);
}
int oracle_getrf_getrs_il_f64(int layout, int n, int nrhs, int64_t batch, int64_t w, double* A,
                              double* B, int32_t* ipiv, int32_t* info, int32_t* tie_step,
                              double tau, int ruda, int scale, int nthreads) {
  return getrf_getrs_il_batched<double>(layout, n, nrhs, batch, w, A, B, ipiv, info, tie_step,
                                     tau, ruda, scale, nthreads);
}
int oracle_potrf_potrs_il_f32(int layout, int fill, int n, int nrhs, int64_t batch, int64_t w,
                              float* A, float* B, int32_t* info, int ruda, int nthreads) {
  return potrf_potrs_il_batched<float>(layout, fill, n, nrhs, batch, w, A, B, info, ruda,
                                     nthreads);
}
int oracle_potrf_potrs_il_f64(int layout, int fill, int n, int nrhs, int64_t batch, int64_t w,
                              double* A, double* B, int32_t* info, int ruda, int nthreads) {
  return potrf_potrs_il_batched<double>(layout, fill, n, nrhs, batch, w, A, B, info, ruda,
                                     nthreads);
}

int oracle_getrf_getrs_mirror_ex_f32(int layout, int n, int nrhs, int64_t batch, int64_t w,
                                     float* A, float* B, int32_t* ipiv, int32_t* info,
                                     int32_t* tie_step, double tau, int scale, int nthreads) {
  return getrf_getrs_mirror_batched<float>(layout, n, nrhs, batch, A, B, ipiv, info, tie_step, tau,
                                         nthreads, w, scale);
}
int oracle_getrf_getrs_mirror_ex_f64(int layout, int n, int nrhs, int64_t batch, int64_t w,
                                     double* A, double* B, int32_t* ipiv, int32_t* info,
                                     int32_t* tie_step, double tau, int scale, int nthreads) {
  return getrf_getrs_mirror_batched<double>(layout, n, nrhs, batch, A, B, ipiv, info, tie_step,
                                          tau, nthreads, w, scale);
}
int oracle_getrf_il_f32(int layout, int n, int64_t batch, int64_t w, float* A, int32_t* ipiv,
                        int32_t* info, int32_t* tie_step, int nthreads) {
  return getrf_il_batched<float>(layout, n, batch, w, A, ipiv, info, tie_step, nthreads);
}
int oracle_getrf_il_f64(int layout, int n, int64_t batch, int64_t w, double* A, int32_t* ipiv,
                        int32_t* info, int32_t* tie_step, int nthreads) {
  return getrf_il_batched<double>(layout, n, batch, w, A, ipiv, info, tie_step, nthreads);
}
int oracle_getrs_il_f32(int layout, int n, int nrhs, int64_t batch, int64_t w, const float* LU,
                        const int32_t* ipiv, float* B, int nthreads) {
  return getrs_il_batched<float>(layout, n, nrhs, batch, w, LU, ipiv, B, nthreads);
}
int oracle_getrs_il_f64(int layout, int n, int nrhs, int64_t batch, int64_t w, const double* LU,
                        const int32_t* ipiv, double* B, int nthreads) {
  return getrs_il_batched<double>(layout, n, nrhs, batch, w, LU, ipiv, B, nthreads);
}
int oracle_potrf_il_f32(int layout, int fill, int n, int64_t batch, int64_t w, float* A,
                        int32_t* info, int nthreads) {
  return potrf_il_batched<float>(layout, fill, n, batch, w, A, info, nthreads);
}
int oracle_potrf_il_f64(int layout, int fill, int n, int64_t batch, int64_t w, double* A,
                        int32_t* info, int nthreads) {
  return potrf_il_batched<double>(layout, fill, n, batch, w, A, info, nthreads);
}
int oracle_potrs_il_f32(int layout, int fill, int n, int nrhs, int64_t batch, int64_t w,
                        const float* L, float* B, int nthreads) {
  return potrs_il_batched<float>(layout, fill, n, nrhs, batch, w, L, B, nthreads);
}
int oracle_potrs_il_f64(int layout, int fill, int n, int nrhs, int64_t batch, int64_t w,
                        const double* L, double* B, int nthreads) {
  return potrs_il_batched<double>(layout, fill, n, nrhs, batch, w, L, B, nthreads);
}

}  // extern "C"
