"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each pin takes an ``oracle.Oracle`` instance, so that the same checks run on the real
oracle (test_oracle_pins.py) and on deliberately broken copies of it
(test_oracle_mutations.py, which shows that every planted mistake trips a pin).
A pin raises AssertionError on failure. None of them calls the CUDA library.

What each pin rests on:
  * closed forms of 2x2 / 3x3 systems worked by hand (exact binary values);
  * Cramer's rule with determinants by permutation expansion in exact rational
    arithmetic, on n <= 4 (brute force);
  * reconstructions P A = L U and A = L L^T;
  * LAPACK (through SciPy) as a library special case: same pivot sequence as dgetrf on
    inputs without near ties, same first failing minor as dpotrf;
  * the info contract on constructed singular / indefinite inputs;
  * the block-tridiagonal solve against dense Cholesky of the assembled matrix;
  * the factor/solve split against the fused routines (same operations, same order),
    a swap-only solve, Cramer's rule and a diagonal factor worked by hand;
  * the block-tridiagonal matvec against integer arithmetic (exact) and the assembled
    dense product.
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np
import scipy.linalg as sla

from gen.workloads import (COL_MAJOR, ROW_MAJOR, assemble_bdsv_dense, deinterleave, from_storage,
                           interleave, to_storage)
from tests.numerics import backward_error, eps_of, forward_error, lapack_perm, unpack_lu


# ----------------------------------------------------------------------------- helpers
def _lu(orc, A_logical, B_logical, layout=ROW_MAJOR):
    A = to_storage(np.asarray(A_logical), layout)
    B = to_storage(np.asarray(B_logical, A.dtype), layout)
    LU, X, ipiv, info, tie = orc.getrf_getrs(A, B, layout)
    return from_storage(LU, layout), from_storage(X, layout), ipiv, info, tie


def _chol(orc, A_logical, B_logical, layout=COL_MAJOR):
    A = to_storage(np.asarray(A_logical), layout)
    B = to_storage(np.asarray(B_logical, A.dtype), layout)
    L, X, info = orc.potrf_potrs(A, B, layout)
    return from_storage(L, layout), from_storage(X, layout), info


def _det_exact(M):
    n = len(M)
    total = Fraction(0)
    for perm in itertools.permutations(range(n)):
        inv = sum(1 for i in range(n) for j in range(i + 1, n) if perm[i] > perm[j])
        term = Fraction(1)
        for i in range(n):
            term *= M[i][perm[i]]
        total += -term if inv % 2 else term
    return total


def _cramer_exact(A, b):
    n = A.shape[0]
    M = [[Fraction(float(A[i, j])) for j in range(n)] for i in range(n)]
    bb = [Fraction(float(v)) for v in b]
    d = _det_exact(M)
    if d == 0:
        return None, d
    xs = []
    for j in range(n):
        Mj = [row[:] for row in M]
        for i in range(n):
            Mj[i][j] = bb[i]
        xs.append(_det_exact(Mj) / d)
    return xs, d


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------------- LU pins
def pin_lu_3x3_hand_worked(orc):
    """Hand-worked 3x3 with a pivot tie at step 2 (lowest-row rule keeps the row).

    A = [[2,1,1],[4,-6,0],[-2,7,2]], b = [5,-2,9]. Step 1 pivots on row 2 (|4|);
    the Schur complement's first column is [4, 4]: a tie, the row in place wins.
    Exact: ipiv = [2,2,3], U = [[4,-6,0],[0,4,1],[0,0,1]], L = [[1],[.5,1],[-.5,1,1]],
    x = [1,1,2]."""
    for dt in (np.float64, np.float32):
        for layout in (ROW_MAJOR, COL_MAJOR):
            A = np.array([[[2, 1, 1], [4, -6, 0], [-2, 7, 2]]], dt)
            b = np.array([[[5], [-2], [9]]], dt)
            LU, X, ipiv, info, _ = _lu(orc, A, b, layout)
            assert info[0] == 0
            assert list(ipiv[0]) == [2, 2, 3], ipiv
            exp = np.array([[4, -6, 0], [0.5, 4, 1], [-0.5, 1, 1]], dt)
            assert np.array_equal(LU[0], exp), LU[0]
            assert np.array_equal(X[0, :, 0], np.array([1, 1, 2], dt)), X


def pin_lu_2x2_closed_form(orc):
    """2x2: the pivot is the larger of |a11|, |a21|; x by Cramer's rule."""
    rng = _rng(11)
    for dt in (np.float64, np.float32):
        eps = eps_of(dt)
        for _ in range(50):
            A = rng.uniform(-1, 1, (2, 2)).astype(dt)
            b = rng.uniform(-1, 1, (2, 1)).astype(dt)
            det = float(A[0, 0]) * float(A[1, 1]) - float(A[0, 1]) * float(A[1, 0])
            if abs(det) < 0.1:
                continue
            LU, X, ipiv, info, _ = _lu(orc, A[None], b[None])
            swap = abs(A[1, 0]) > abs(A[0, 0])
            assert list(ipiv[0]) == ([2, 2] if swap else [1, 2])
            a = A.astype(np.float64)
            if swap:
                a = a[::-1]
                bb = b.astype(np.float64)[::-1]
            else:
                bb = b.astype(np.float64)
            l21 = a[1, 0] / a[0, 0]
            u22 = a[1, 1] - l21 * a[0, 1]
            exp = np.array([[a[0, 0], a[0, 1]], [l21, u22]])
            assert np.allclose(LU[0], exp, rtol=8 * eps, atol=8 * eps), (LU[0], exp)
            x1 = (float(b[0, 0]) * float(A[1, 1]) - float(A[0, 1]) * float(b[1, 0])) / det
            x2 = (float(A[0, 0]) * float(b[1, 0]) - float(b[0, 0]) * float(A[1, 0])) / det
            kappa = np.linalg.cond(a)
            tol = 16 * kappa * eps
            assert np.allclose(X[0, :, 0], [x1, x2], rtol=tol, atol=tol), (X[0, :, 0], x1, x2)
            del bb


def pin_lu_cramer_bruteforce(orc):
    """n <= 4: the oracle's x against the exact rational solution (Cramer, Leibniz
    determinants), and prod(diag U) * (-1)^swaps against the exact determinant."""
    rng = _rng(12)
    for dt in (np.float64, np.float32):
        eps = eps_of(dt)
        for n in (1, 2, 3, 4):
            for _ in range(12):
                A = rng.integers(-9, 10, (n, n)).astype(dt)
                b = rng.integers(-9, 10, (n, 1)).astype(dt)
                xs, d = _cramer_exact(A, b[:, 0])
                if d == 0:
                    continue
                LU, X, ipiv, info, _ = _lu(orc, A[None], b[None])
                assert info[0] == 0
                kappa = np.linalg.cond(A.astype(np.float64))
                xe = np.array([float(v) for v in xs])
                err = np.abs(X[0, :, 0].astype(np.float64) - xe).max() / max(np.abs(xe).max(), 1e-300)
                assert err <= 8 * n * kappa * eps, (n, err, kappa)
                swaps = sum(1 for k in range(n) if ipiv[0, k] != k + 1)
                detu = float(np.prod(np.diag(LU[0]).astype(np.float64))) * (-1) ** swaps
                assert abs(detu - float(d)) <= 8 * n * eps * max(abs(float(d)), 1.0) * kappa, (detu, d)


def pin_lu_reconstruction(orc):
    """P A = L U to within a small multiple of n eps ||A|| (both dtypes, both layouts)."""
    rng = _rng(13)
    for dt in (np.float64, np.float32):
        eps = eps_of(dt)
        for n in (1, 3, 8, 16, 33):
            A = rng.standard_normal((6, n, n)).astype(dt)
            B = rng.standard_normal((6, n, 2)).astype(dt)
            for layout in (ROW_MAJOR, COL_MAJOR):
                LU, X, ipiv, info, _ = _lu(orc, A, B, layout)
                for s in range(A.shape[0]):
                    L, U = unpack_lu(LU[s])
                    P = lapack_perm(ipiv[s])
                    res = np.abs(A[s].astype(np.float64)[P] - L @ U).max()
                    assert res <= 4 * n * eps * np.abs(A[s]).max(), (n, res)


def pin_lu_matches_lapack(orc):
    """Against LAPACK dgetrf/sgetrf (SciPy): identical pivot sequence on inputs without
    near ties, factors and solutions to rounding."""
    rng = _rng(14)
    for dt in (np.float64, np.float32):
        eps = eps_of(dt)
        for n in (2, 5, 16, 32, 64):
            A = rng.standard_normal((5, n, n)).astype(dt)
            B = rng.standard_normal((5, n, 3)).astype(dt)
            LU, X, ipiv, info, tie = _lu(orc, A, B)
            for s in range(A.shape[0]):
                lu, piv = sla.lu_factor(A[s])
                if tie[s] < 0:
                    assert np.array_equal(piv + 1, ipiv[s]), (piv + 1, ipiv[s])
                    assert np.allclose(LU[s], lu, rtol=0, atol=64 * n * eps * np.abs(lu).max())
                be = backward_error(A[s][None], X[s][None], B[s][None])[0]
                assert be <= 8 * n * eps, be


def pin_lu_info_contract(orc):
    """info = first singular pivot (1-based); X = 0; ipiv still reported.

    * column j zeroed: the column stays exactly zero, the tie among zeros keeps the row
      in place: info = j + 1, ipiv[j] = j + 1;
    * [[1,2],[2,4]]: pivot 2, then 4 - 0.5*... = 0 exactly: info = 2;
    * 1x1 subnormal pivot is singular, the smallest normal is not (singular floor)."""
    rng = _rng(15)
    for dt in (np.float64, np.float32):
        n = 8
        for j in range(n):
            A = rng.uniform(-1, 1, (1, n, n)).astype(dt)
            A[0, :, j] = 0
            b = rng.uniform(-1, 1, (1, n, 1)).astype(dt)
            LU, X, ipiv, info, _ = _lu(orc, A, b)
            assert info[0] == j + 1, (j, info)
            assert ipiv[0, j] == j + 1
            assert np.all(X == 0)
        LU, X, ipiv, info, _ = _lu(orc, np.array([[[1, 2], [2, 4]]], dt), np.ones((1, 2, 1), dt))
        assert info[0] == 2 and list(ipiv[0]) == [2, 2] and np.all(X == 0)
        tiny = np.finfo(dt).smallest_subnormal
        _, X, _, info, _ = _lu(orc, np.array([[[tiny]]], dt), np.ones((1, 1, 1), dt))
        assert info[0] == 1 and X[0, 0, 0] == 0
        _, X, _, info, _ = _lu(orc, np.array([[[np.finfo(dt).tiny]]], dt), np.ones((1, 1, 1), dt))
        assert info[0] == 0 and X[0, 0, 0] == dt(1) / np.finfo(dt).tiny
        # only the first failing pivot is reported
        A = np.zeros((1, 3, 3), dt)
        A[0, 2, 2] = 1
        _, _, ipiv, info, _ = _lu(orc, A, np.ones((1, 3, 1), dt))
        assert info[0] == 1 and list(ipiv[0]) == [1, 2, 3]


def pin_lu_layout_invariance(orc):
    """Row- and column-major storage of the same A give the same pivots, info and,
    the arithmetic being identical, bitwise identical factors and solutions."""
    rng = _rng(16)
    for dt in (np.float64, np.float32):
        A = rng.standard_normal((10, 12, 12)).astype(dt)
        B = rng.standard_normal((10, 12, 3)).astype(dt)
        r = _lu(orc, A, B, ROW_MAJOR)
        c = _lu(orc, A, B, COL_MAJOR)
        for a, b in zip(r, c):
            assert np.array_equal(a, b)


def pin_lu_near_tie_flag(orc):
    """The near-tie record: two top candidates within 1e-6 relative at step 0."""
    A = np.array([[[1.0, 2.0], [1.0 + 1e-9, 3.0]]])
    _, _, _, _, tie = _lu(orc, A, np.ones((1, 2, 1)))
    assert tie[0] == 0
    A = np.array([[[1.0, 2.0], [0.5, 3.0]]])
    _, _, _, _, tie = _lu(orc, A, np.ones((1, 2, 1)))
    assert tie[0] == -1


# ----------------------------------------------------------------------- Cholesky pins
def pin_chol_hand_worked(orc):
    """A = L L^T with L = [[2,0,0],[1,3,0],[-1,2,4]]: A = [[4,2,-2],[2,10,5],[-2,5,21]];
    with b = A [1,1,1]^T = [4,17,24] the solution is [1,1,1]."""
    for dt in (np.float64, np.float32):
        eps = eps_of(dt)
        for layout in (COL_MAJOR, ROW_MAJOR):
            A = np.array([[[4, 2, -2], [2, 10, 5], [-2, 5, 21]]], dt)
            b = np.array([[[4], [17], [24]]], dt)
            L, X, info = _chol(orc, A, b, layout)
            assert info[0] == 0
            Lexp = np.array([[2, 0, 0], [1, 3, 0], [-1, 2, 4]], np.float64)
            assert np.allclose(np.tril(L[0]), Lexp, rtol=0, atol=8 * eps * 4)
            assert np.allclose(X[0, :, 0], [1, 1, 1], rtol=0, atol=64 * eps)


def pin_chol_2x2_closed_form(orc):
    """l11 = sqrt(a11), l21 = a21 / l11, l22 = sqrt(a22 - l21^2)."""
    rng = _rng(21)
    for dt in (np.float64, np.float32):
        eps = eps_of(dt)
        for _ in range(40):
            G = rng.standard_normal((2, 2))
            A = (G @ G.T + 0.5 * np.eye(2)).astype(dt)
            L, X, info = _chol(orc, A[None], np.ones((1, 2, 1), dt))
            a = A.astype(np.float64)
            l11 = np.sqrt(a[0, 0])
            l21 = a[1, 0] / l11
            l22 = np.sqrt(a[1, 1] - l21 * l21)
            assert info[0] == 0
            assert np.allclose([L[0, 0, 0], L[0, 1, 0], L[0, 1, 1]], [l11, l21, l22],
                               rtol=16 * eps * np.linalg.cond(a), atol=0)


def pin_chol_reconstruction_and_lapack(orc):
    """A = L L^T; L against LAPACK dpotrf; x against the exact rational solution for
    n <= 4 integer SPD matrices; only the lower triangle is written."""
    rng = _rng(22)
    for dt in (np.float64, np.float32):
        eps = eps_of(dt)
        for n in (1, 4, 9, 32):
            G = rng.standard_normal((4, n, n))
            A = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dt)
            B = rng.standard_normal((4, n, 2)).astype(dt)
            for layout in (COL_MAJOR, ROW_MAJOR):
                L, X, info = _chol(orc, A, B, layout)
                assert np.all(info == 0)
                for s in range(4):
                    Ls = np.tril(L[s]).astype(np.float64)
                    assert np.abs(Ls @ Ls.T - A[s]).max() <= 4 * n * eps * np.abs(A[s]).max()
                    ref = sla.cholesky(A[s].astype(np.float64), lower=True)
                    assert np.allclose(Ls, ref, rtol=0, atol=32 * n * eps * np.abs(ref).max())
                    # the strictly upper triangle is untouched
                    iu = np.triu_indices(n, 1)
                    assert np.array_equal(L[s][iu], A[s][iu])
                be = backward_error(A, X, B)
                assert np.all(be <= 8 * n * eps), be
        for n in (2, 3, 4):
            for _ in range(6):
                G = rng.integers(-3, 4, (n, n))
                A = (G @ G.T + np.eye(n, dtype=int)).astype(dt)
                b = rng.integers(-5, 6, (n, 1)).astype(dt)
                xs, d = _cramer_exact(A, b[:, 0])
                _, X, info = _chol(orc, A[None], b[None])
                xe = np.array([float(v) for v in xs])
                kappa = np.linalg.cond(A.astype(np.float64))
                err = np.abs(X[0, :, 0] - xe).max() / max(np.abs(xe).max(), 1e-300)
                assert err <= 16 * n * kappa * eps, (err, kappa)


def pin_chol_info_contract(orc):
    """info = smallest leading minor that is not positive definite; X = 0.

    * A[k][k] = -1 on an SPD matrix (minors 1..k untouched, the (k+1)-th Schur value
      is <= -1): info = k + 1;
    * agreement with LAPACK dpotrf's info on random indefinite matrices;
    * a zero or NaN diagonal fails (!(d > 0))."""
    rng = _rng(23)
    for dt in (np.float64, np.float32):
        n = 12
        for k in range(n):
            G = rng.standard_normal((n, n))
            A = (G @ G.T + n * np.eye(n)).astype(dt)
            A[k, k] = -1
            _, X, info = _chol(orc, A[None], np.ones((1, n, 1), dt))
            assert info[0] == k + 1 and np.all(X == 0)
        for _ in range(20):
            S = rng.standard_normal((n, n))
            A = ((S + S.T) / 2 + rng.uniform(-1, 4) * np.eye(n)).astype(dt)
            _, _, info = _chol(orc, A[None], np.ones((1, n, 1), dt))
            potrf = sla.lapack.dpotrf if dt == np.float64 else sla.lapack.spotrf
            _, linfo = potrf(A, lower=1)
            assert info[0] == linfo, (info[0], linfo)
        A = np.diag([1.0, 0.0, 1.0]).astype(dt)
        assert _chol(orc, A[None], np.ones((1, 3, 1), dt))[2][0] == 2
        A = np.diag([1.0, 1.0, np.nan]).astype(dt)
        assert _chol(orc, A[None], np.ones((1, 3, 1), dt))[2][0] == 3


def pin_chol_upper_fill(orc):
    """Upper fill (cuSolverDx POTRF: A = U^T U, only the upper triangle processed and
    replaced by U, the lower part untouched): the 2x2 closed form u11 = sqrt(a11),
    u12 = a12/u11, u22 = sqrt(a22 - u12^2); U^T U = A to rounding; U equals the
    transpose of the lower factor of the same matrix (the Cholesky factor is unique);
    NaN in the lower triangle is never read; a planted indefinite minor gives the same
    info as lower fill; the solve meets the backward-error bound."""
    A2 = np.array([[[4.0, 2.0], [np.nan, 5.0]]])          # upper fill, row-major
    U, X, info = orc.potrf_potrs(A2, np.array([[[8.0], [9.0]]]), ROW_MAJOR, fill=1)
    assert info[0] == 0 and U[0, 0, 0] == 2.0 and U[0, 0, 1] == 1.0 and U[0, 1, 1] == 2.0
    assert np.isnan(U[0, 1, 0])
    assert np.allclose(X[0, :, 0], [1.375, 1.25], rtol=0, atol=1e-15)
    rng = _rng(28)
    for dt in (np.float64, np.float32):
        eps = eps_of(dt)
        for layout in (ROW_MAJOR, COL_MAJOR):
            for n in (1, 5, 17, 40):
                G = rng.standard_normal((4, n, n))
                Al = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dt)
                if n > 2:
                    Al[2, n // 2, n // 2] = -1.0
                B = rng.standard_normal((4, n, 2)).astype(dt)
                Au = Al.copy()
                Al_ = Al.copy()
                il, iu = np.tril_indices(n, -1), np.triu_indices(n, 1)
                Au[:, il[0], il[1]] = np.nan
                Al_[:, iu[0], iu[1]] = np.nan
                Uu, Xu, infu = orc.potrf_potrs(to_storage(Au, layout), to_storage(B, layout), layout, fill=1)
                Ll, Xl, infl = orc.potrf_potrs(to_storage(Al_, layout), to_storage(B, layout), layout, fill=0)
                Uu, Ll = from_storage(Uu, layout), from_storage(Ll, layout)
                Xu, Xl = from_storage(Xu, layout), from_storage(Xl, layout)
                assert np.array_equal(infu, infl)
                assert np.all(np.isnan(Uu[:, il[0], il[1]]))
                ok = infu == 0
                assert np.array_equal(np.triu(np.nan_to_num(Uu[ok])),
                                      np.swapaxes(np.tril(np.nan_to_num(Ll[ok])), 1, 2))
                assert np.array_equal(Xu[ok], Xl[ok])
                Ut = np.triu(np.nan_to_num(Uu[ok])).astype(np.float64)
                Asym = np.triu(Al[ok]) + np.swapaxes(np.triu(Al[ok], 1), 1, 2)
                rec = np.swapaxes(Ut, 1, 2) @ Ut
                assert np.allclose(rec, Asym, rtol=0, atol=16 * n * eps * np.abs(Asym).max())
                be = backward_error(Asym, Xu[ok], B[ok])
                assert np.all(be <= 8 * n * eps)


# ----------------------------------------------------------------- contract variants
def pin_threshold_pivoting(orc):
    """TDLS threshold pivoting (relative_pivot_threshold tau): tau = 1 is partial pivoting
    bit for bit; the hand-worked 2x2 [[0.6, 1], [1, 1]] keeps its first row for tau = 0.5
    (0.6 >= 0.5 * 1) and swaps for tau = 0.7; on random matrices every multiplier obeys
    |l_ik| <= 1/tau (the growth bound threshold pivoting exists for) and P A = L U holds to
    rounding."""
    rng = _rng(51)
    for dt in (np.float32, np.float64):
        for layout in (ROW_MAJOR, COL_MAJOR):
            A = rng.standard_normal((6, 9, 9)).astype(dt)
            A[2, :, 4] = 0
            B = rng.standard_normal((6, 9, 2)).astype(dt)
            As, Bs = to_storage(A, layout), to_storage(B, layout)
            r1 = orc.getrf_getrs(As, Bs, layout)
            r2 = orc.getrf_getrs_ex(As, Bs, layout, tau=1.0)
            assert all(np.array_equal(x, y) for x, y in zip(r1, r2))
    A2 = np.array([[[0.6, 1.0], [1.0, 1.0]]])
    b2 = np.array([[[1.0], [2.0]]])
    LU, X, ipiv, info, _ = orc.getrf_getrs_ex(A2, b2, ROW_MAJOR, tau=0.5)
    assert list(ipiv[0]) == [1, 2] and LU[0, 0, 0] == 0.6 and info[0] == 0
    assert np.allclose(X[0, :, 0], np.linalg.solve(A2[0], b2[0, :, 0]), rtol=1e-14)
    LU, X, ipiv, info, _ = orc.getrf_getrs_ex(A2, b2, ROW_MAJOR, tau=0.7)
    assert list(ipiv[0]) == [2, 2] and LU[0, 0, 0] == 1.0
    # the kept pivot is judged by its own magnitude: 0.9 * FLT_MIN (subnormal) stays in
    # place against FLT_MIN with tau = 0.5, and is singular (info = 1)
    fmin = np.finfo(np.float32).tiny
    A3 = np.array([[[0.9 * fmin, 1.0], [fmin, 1.0]]], np.float32)
    LU, X, ipiv, info, _ = orc.getrf_getrs_ex(A3, np.ones((1, 2, 1), np.float32), ROW_MAJOR, tau=0.5)
    assert ipiv[0, 0] == 1 and info[0] == 1
    for tau in (0.1, 0.5, 0.9):
        A = rng.standard_normal((20, 12, 12))
        B = rng.standard_normal((20, 12, 1))
        LU, X, ipiv, info, tie = orc.getrf_getrs_ex(A, B, ROW_MAJOR, tau=tau)
        for s in range(20):
            L, U = unpack_lu(LU[s])
            assert np.abs(L).max() <= (1.0 / tau) * (1 + 1e-12)
            PA = A[s][lapack_perm(ipiv[s])]
            growth = max(np.abs(U).max() / np.abs(A[s]).max(), 1.0)
            err = np.abs(PA - L @ U).max() / np.abs(A[s]).max()
            assert err <= 64 * 12 * eps_of(np.float64) * growth, (tau, s, err)


def pin_ruda_status_lu(orc):
    """RUDA status contract on constructed inputs: a NaN in A or an inf in B gives -1; a
    zero column j gives j + 1; a finite input whose solution overflows (FP32 diag(1e-30, 1),
    b = (1e10, 1): x_0 = 1e40) gives -3; each failed system returns zeros and ipiv = -1;
    a system that succeeds is the default contract's bit for bit."""
    n = 4
    rng = _rng(52)
    A = rng.standard_normal((5, n, n)).astype(np.float32) + 3 * np.eye(n, dtype=np.float32)
    B = rng.standard_normal((5, n, 1)).astype(np.float32)
    A[0, 1, 2] = np.nan
    B[1, 3, 0] = np.inf
    A[2, :, 1] = 0
    A[3] = np.diag([1e-30, 1.0, 1.0, 1.0]).astype(np.float32)
    B[3, :, 0] = [1e10, 1.0, 1.0, 1.0]
    LU, X, ipiv, info, _ = orc.getrf_getrs_ex(A, B, ROW_MAJOR, ruda=1)
    assert list(info) == [-1, -1, 2, -3, 0], info
    for s in range(4):
        assert np.all(LU[s] == 0) and np.all(X[s] == 0) and np.all(ipiv[s] == -1)
    d = orc.getrf_getrs(A[4:], B[4:], ROW_MAJOR)
    assert np.array_equal(LU[4], d[0][0]) and np.array_equal(X[4], d[1][0])
    assert np.array_equal(ipiv[4], d[2][0])


def pin_ruda_status_chol(orc):
    """RUDA status contract for Cholesky: NaN in A or inf in B -> -1; one off-diagonal pair
    differing in its last bit -> -2 (the symmetry check is exact); A[k][k] = -1 -> k + 1; FP32
    diag(1e-30, ...) with b = 1e30 overflows y -> -3; failures return the factor's
    triangle and X as zeros; a success is the default contract's bit for bit."""
    n = 5
    rng = _rng(53)
    G = rng.standard_normal((5, n, n))
    A = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(np.float32)
    B = rng.standard_normal((5, n, 2)).astype(np.float32)
    A = np.concatenate([A, A[4:]])       # system 5: a copy of the good one with inf in B
    B = np.concatenate([B, B[4:]])
    B[5, 2, 1] = np.inf
    A[0, 3, 3] = np.nan
    A[1, 1, 3] = np.nextafter(A[1, 1, 3], np.float32(np.inf))
    A[2, 2, 2] = -1.0
    A[3] = np.diag([1e-30] * n).astype(np.float32)
    B[3] = 1e30
    for fill in (0, 1):
        L, X, info = orc.potrf_potrs_ex(A, B, ROW_MAJOR, fill=fill, ruda=1)
        assert list(info) == [-1, -2, 3, -3, 0, -1], (fill, info)
        tri = np.tril_indices(n) if fill == 0 else np.triu_indices(n)
        for s in (0, 1, 2, 3, 5):
            assert np.all(L[s][tri] == 0) and np.all(X[s] == 0)
        d = orc.potrf_potrs(A[4:5], B[4:5], ROW_MAJOR, fill=fill)
        assert np.array_equal(L[4], d[0][0]) and np.array_equal(X[4], d[1][0])


def pin_tdls_row_major_reading(orc):
    """TDLS row-major reading (P A^T = L U, A = U^T L^T P): the hand-worked 2x2 A =
    [[1, 2], [3, 4]] factors S = A^T = [[1, 3], [2, 4]] with ipiv = (2, 2), L = [[1, 0],
    [0.5, 1]], U = [[2, 4], [0, 1]], stored back through the column-major reading as rows
    (2, 0.5) and (4, 1); b = (5, 6) gives x = (-4, 4.5) exactly. On random systems the
    factor is the default factor of the memory read column-major (bit for bit), the
    solution meets the backward-error bound, and column-major storage is the default
    path."""
    A = np.array([[[1.0, 2.0], [3.0, 4.0]]])
    b = np.array([[[5.0], [6.0]]])
    S, X, ipiv, info, _ = orc.getrf_getrs_mirror(A, b, ROW_MAJOR)
    assert list(ipiv[0]) == [2, 2] and info[0] == 0
    assert np.array_equal(S[0], [[2.0, 0.5], [4.0, 1.0]])
    assert np.array_equal(X[0, :, 0], [-4.0, 4.5])
    rng = _rng(54)
    for dt in (np.float32, np.float64):
        n = 13
        A = rng.standard_normal((8, n, n)).astype(dt)
        B = rng.standard_normal((8, n, 3)).astype(dt)
        A[2, 4, :] = 0                   # a zero row of A: a zero column of S
        S, X, ipiv, info, _ = orc.getrf_getrs_mirror(A, B, ROW_MAJOR)
        S2, ip2, inf2, _ = orc.getrf(A, COL_MAJOR)
        assert np.array_equal(S, S2) and np.array_equal(ipiv, ip2) and np.array_equal(info, inf2)
        assert info[2] > 0 and np.all(X[2] == 0)
        ok = info == 0
        be = backward_error(A[ok].astype(np.float64), X[ok], B[ok])
        assert np.all(be <= 8 * n * eps_of(dt))
        Ac = to_storage(A, COL_MAJOR)
        Bc = to_storage(B, COL_MAJOR)
        r1 = orc.getrf_getrs_mirror(Ac, Bc, COL_MAJOR)
        r2 = orc.getrf_getrs(Ac, Bc, COL_MAJOR)
        assert all(np.array_equal(x, y) for x, y in zip(r1, r2))


# --------------------------------------------------------------------------- bdsv pins
def _random_bdsv(rng, batch, nbr, bs, dt=np.float64):
    strips = np.zeros((batch, nbr, bs, 3 * bs), dt)
    C = rng.uniform(-0.5, 0.5, (batch, max(nbr - 1, 0), bs, bs)) / bs
    M = rng.standard_normal((batch, nbr, bs, bs)) / np.sqrt(bs)
    strips[:, :, :, bs:2 * bs] = M @ np.swapaxes(M, 2, 3) + 3.0 * np.eye(bs)
    if nbr > 1:
        strips[:, :nbr - 1, :, 2 * bs:] = C
        strips[:, 1:, :, :bs] = np.swapaxes(C, 2, 3)
    xpad = np.zeros((batch, (nbr + 2) * bs), dt)
    xpad[:, bs:(nbr + 1) * bs] = rng.standard_normal((batch, nbr * bs))
    return strips, xpad


def pin_bdsv_dense_equivalence(orc):
    """bdsv equals the dense solve of the assembled matrix (backward error), its MAIN
    blocks are the diagonal blocks of the dense Cholesky factor and its LEFT blocks the
    sub-diagonal ones; RIGHT slots, the upper triangles of MAIN and the pads are left as
    they were."""
    rng = _rng(31)
    for dt in (np.float64, np.float32):
        eps = eps_of(dt)
        for nbr, bs in ((1, 4), (2, 3), (5, 8), (32, 8)):
            strips, xpad = _random_bdsv(rng, 3, nbr, bs, dt)
            S, X, info = orc.bdsv(strips, xpad)
            assert np.all(info == 0)
            Ad = assemble_bdsv_dense(strips).astype(np.float64)
            N = nbr * bs
            b = xpad[:, bs:bs + N]
            x = X[:, bs:bs + N]
            be = backward_error(Ad, x[:, :, None], b[:, :, None])
            assert np.all(be <= 8 * N * eps), be
            for s in range(3):
                Lf = np.linalg.cholesky(Ad[s])
                for k in range(nbr):
                    r0 = k * bs
                    F = np.tril(S[s, k, :, bs:2 * bs])
                    assert np.allclose(F, Lf[r0:r0 + bs, r0:r0 + bs], rtol=0, atol=64 * N * eps)
                    iu = np.triu_indices(bs, 1)
                    assert np.array_equal(S[s, k, :, bs:2 * bs][iu], strips[s, k, :, bs:2 * bs][iu])
                    if k > 0:
                        assert np.allclose(S[s, k, :, :bs], Lf[r0:r0 + bs, r0 - bs:r0], rtol=0,
                                           atol=64 * N * eps)
                assert np.array_equal(S[s, :, :, 2 * bs:], strips[s, :, :, 2 * bs:])
                assert np.all(X[s, :bs] == 0) and np.all(X[s, bs + N:] == 0)


def pin_bdsv_single_block_is_potrf(orc):
    """NBR = 1 reduces to Cholesky factor + solve of D_0 (LAPACK dpotrf/dpotrs)."""
    rng = _rng(32)
    strips, xpad = _random_bdsv(rng, 4, 1, 6)
    S, X, info = orc.bdsv(strips, xpad)
    for s in range(4):
        D = strips[s, 0, :, 6:12]
        c = sla.cho_factor(D, lower=True)
        x = sla.cho_solve(c, xpad[s, 6:12])
        assert np.allclose(np.tril(S[s, 0, :, 6:12]), np.tril(c[0]), rtol=0, atol=1e-13)
        assert np.allclose(X[s, 6:12], x, rtol=1e-12, atol=1e-14)


def pin_bdsv_scalar_tridiagonal(orc):
    """BS = 1, NBR = 2: [[d0, c], [c, d1]] gives f0 = sqrt(d0), e1 = c / f0,
    f1 = sqrt(d1 - e1^2) (the scalar block-Thomas recurrence)."""
    strips = np.zeros((1, 2, 1, 3))
    d0, d1, c = 4.0, 5.0, 2.0
    strips[0, 0, 0, 1], strips[0, 0, 0, 2] = d0, c
    strips[0, 1, 0, 0], strips[0, 1, 0, 1] = c, d1
    xpad = np.array([[0.0, 8.0, 9.0, 0.0]])
    S, X, info = orc.bdsv(strips, xpad)
    f0 = 2.0
    e1 = 1.0
    f1 = 2.0
    assert S[0, 0, 0, 1] == f0 and S[0, 1, 0, 0] == e1 and S[0, 1, 0, 1] == f1
    # [[4,2],[2,5]] x = [8,9] -> x = [(40-18)/16, (36-16)/16] = [1.375, 1.25]
    assert np.allclose(X[0], [0.0, 1.375, 1.25, 0.0], rtol=0, atol=1e-15)


def pin_bdsv_info(orc):
    """A non-positive-definite knot: info = global index br*bs + j + 1, the same minor
    at which LAPACK dpotrf fails on the assembled dense matrix; X = 0."""
    rng = _rng(33)
    nbr, bs = 6, 4
    for knot in (0, 3, 5):
        for j in (0, 2):
            strips, xpad = _random_bdsv(rng, 1, nbr, bs)
            strips[0, knot, j, bs + j] = -1.0
            S, X, info = orc.bdsv(strips, xpad)
            _, linfo = sla.lapack.dpotrf(assemble_bdsv_dense(strips)[0], lower=1)
            assert info[0] == linfo == knot * bs + j + 1, (info[0], linfo)
            assert np.all(X == 0)


# ----------------------------------------------------- factor once, solve per right-hand side
def pin_getrs_composition(orc):
    """getrf then getrs reproduces the fused getrf+getrs bit for bit (the interchanges
    applied in step order, then each b_i's updates in increasing k, are the fused
    sweep's operations in the fused sweep's order); getrf alone leaves the same
    factor, pivots and info, singular systems included."""
    rng = _rng(41)
    for dt in (np.float32, np.float64):
        for layout in (ROW_MAJOR, COL_MAJOR):
            for n, nrhs in ((1, 1), (3, 2), (8, 1), (16, 4), (33, 3)):
                A = rng.standard_normal((6, n, n)).astype(dt)
                A[1, :, n // 2] = 0        # singular: info > 0
                B = rng.standard_normal((6, n, nrhs)).astype(dt)
                As, Bs = to_storage(A, layout), to_storage(B, layout)
                LU, X, ipiv, info, tie = orc.getrf_getrs(As, Bs, layout)
                LU2, ipiv2, info2, tie2 = orc.getrf(As, layout)
                assert np.array_equal(LU, LU2) and np.array_equal(ipiv, ipiv2)
                assert np.array_equal(info, info2) and np.array_equal(tie, tie2)
                X2 = orc.getrs(LU2, ipiv2, Bs, layout)
                ok = info == 0
                assert np.array_equal(X[ok], X2[ok])


def pin_getrs_permutation_only(orc):
    """With L = U = I the solve is the swap sequence alone: row k of B exchanged with row
    ipiv[k]-1 for k = 0..n-1, in that order (exact); an entry outside 1..n swaps nothing."""
    rng = _rng(42)
    n, nrhs = 6, 3
    LU = np.broadcast_to(np.eye(n), (5, n, n)).copy()
    ipiv = np.stack([rng.integers(k, n, size=5) for k in range(n)], axis=1).astype(np.int32) + 1
    B = rng.standard_normal((5, n, nrhs))
    X = orc.getrs(LU, ipiv, B, ROW_MAJOR)
    for s in range(5):
        want = B[s].copy()
        for k in range(n):
            p = ipiv[s, k] - 1
            want[[k, p]] = want[[p, k]]
        assert np.array_equal(X[s], want)
    # entries outside 1..n swap nothing (the solve reports no status): zero, negative and
    # past-the-end entries leave their rows where they are, in-range ones still swap
    bad = np.array([[0, 3, 7, -2, 6, 2 ** 31 - 1]], np.int32)
    X = orc.getrs(np.eye(n)[None].copy(), bad, B[:1], ROW_MAJOR)
    want = B[0].copy()
    want[[1, 2]] = want[[2, 1]]             # k = 1: row 3
    want[[4, 5]] = want[[5, 4]]             # k = 4: row 6
    assert np.array_equal(X[0], want)


def pin_getrs_cramer(orc):
    """getrf + getrs on n <= 4 agrees with Cramer's rule in exact rational arithmetic
    (determinants by permutation expansion) to a few ulps, for every right-hand side."""
    rng = _rng(43)
    for n in (2, 3, 4):
        A = rng.uniform(-1, 1, (4, n, n))
        B = rng.uniform(-1, 1, (4, n, 2))
        LU, ipiv, info, _ = orc.getrf(A, ROW_MAJOR)
        X = orc.getrs(LU, ipiv, B, ROW_MAJOR)
        for s in range(4):
            for c in range(2):
                xs, d = _cramer_exact(A[s], B[s, :, c])
                assert xs is not None
                want = np.array([float(v) for v in xs])
                assert np.allclose(X[s, :, c], want, rtol=1e-12, atol=1e-13), (X[s, :, c], want)


def pin_potrs_composition(orc):
    """potrf then potrs reproduces the fused potrf+potrs bit for bit; potrf alone leaves
    the same factor and info."""
    rng = _rng(44)
    for dt in (np.float32, np.float64):
        for layout in (ROW_MAJOR, COL_MAJOR):
            for n, nrhs in ((1, 1), (4, 2), (32, 1), (40, 3)):
                G = rng.standard_normal((5, n, n))
                A = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dt)
                A[2, n - 1, n - 1] = -1.0
                B = rng.standard_normal((5, n, nrhs)).astype(dt)
                As, Bs = to_storage(A, layout), to_storage(B, layout)
                L, X, info = orc.potrf_potrs(As, Bs, layout)
                L2, info2 = orc.potrf(As, layout)
                assert np.array_equal(L, L2) and np.array_equal(info, info2)
                X2 = orc.potrs(L2, Bs, layout)
                ok = info == 0
                assert np.array_equal(X[ok], X2[ok])


def pin_potrs_diagonal(orc):
    """L = diag(d): x_i = (b_i * (1/d_i)) * (1/d_i), each product rounded once."""
    d = np.array([[2.0, 0.5, 3.0, 7.0]])
    L = np.zeros((1, 4, 4))
    L[0][np.diag_indices(4)] = d[0]
    b = np.array([[[1.0], [3.0], [5.0], [11.0]]])
    X = orc.potrs(L, b, ROW_MAJOR)
    r = 1.0 / d[0]
    assert np.array_equal(X[0, :, 0], (b[0, :, 0] * r) * r)


def pin_potrs_dense(orc):
    """potrs with a factor from LAPACK dpotrf solves L L^T x = b to the backward-error
    bound (upper triangle of the factor storage ignored)."""
    rng = _rng(45)
    n = 12
    G = rng.standard_normal((3, n, n))
    A = G @ np.swapaxes(G, 1, 2) + n * np.eye(n)
    B = rng.standard_normal((3, n, 2))
    L = np.stack([np.linalg.cholesky(A[s]) for s in range(3)])
    L = L + np.triu(np.full((n, n), 9.0), 1)   # garbage above the diagonal
    X = orc.potrs(to_storage(L, COL_MAJOR), to_storage(B, COL_MAJOR), COL_MAJOR)
    X = from_storage(X, COL_MAJOR)
    be = backward_error(A, X, B)
    assert np.all(be <= 8 * n * eps_of(np.float64)), be


def pin_bdsv_split(orc):
    """bdsv_factor then bdsv_solve reproduces the fused bdsv bit for bit; one factor
    serves several right-hand sides (factor once, solve per right-hand side)."""
    rng = _rng(46)
    for dt in (np.float64, np.float32):
        for nbr, bs in ((1, 3), (4, 5), (32, 8)):
            strips, xpad = _random_bdsv(rng, 3, nbr, bs, dt)
            _, xpad2 = _random_bdsv(rng, 3, nbr, bs, dt)
            S, X, info = orc.bdsv(strips, xpad)
            S2, info2 = orc.bdsv_factor(strips)
            assert np.array_equal(S, S2) and np.array_equal(info, info2)
            assert np.array_equal(orc.bdsv_solve(S2, xpad), X)
            _, Xb, _ = orc.bdsv(strips, xpad2)
            assert np.array_equal(orc.bdsv_solve(S2, xpad2), Xb)


# --------------------------------------------------------------------------- bdmv pins
def pin_bdmv_exact_integers(orc):
    """Small integers make every product and partial sum exact, so y must equal the
    window definition evaluated in integers: y[(br+1)bs + r] = sum over the strip row of
    strip[br][r][c] * x[br*bs + c]; the pad blocks of y keep their input values."""
    rng = _rng(47)
    for nbr, bs in ((1, 2), (3, 4), (5, 8)):
        strips = rng.integers(-9, 10, (2, nbr, bs, 3 * bs)).astype(np.float64)
        xpad = rng.integers(-9, 10, (2, (nbr + 2) * bs)).astype(np.float64)
        xpad[:, :bs] = 0
        xpad[:, (nbr + 1) * bs:] = 0
        ypad = np.full_like(xpad, 7.0)
        Y = orc.bdmv(strips, xpad, ypad)
        for s in range(2):
            Si = strips[s].astype(np.int64)
            xi = xpad[s].astype(np.int64)
            for br in range(nbr):
                for r in range(bs):
                    want = int(sum(int(Si[br, r, c]) * int(xi[br * bs + c]) for c in range(3 * bs)))
                    assert Y[s, (br + 1) * bs + r] == want
            assert np.all(Y[s, :bs] == 7.0) and np.all(Y[s, (nbr + 1) * bs:] == 7.0)


def pin_bdmv_dense(orc):
    """y agrees with the assembled dense matrix times x (NumPy, float64) within the dot
    product rounding bound gamma_{3bs} |A| |x|; the edge blocks L_0 / R_{nbr-1} multiply
    the zero pads."""
    rng = _rng(48)
    for dt in (np.float64, np.float32):
        eps = eps_of(dt)
        for nbr, bs in ((1, 4), (6, 3), (32, 8)):
            strips, xpad = _random_bdsv(rng, 3, nbr, bs, dt)
            strips[:, 0, :, :bs] = rng.standard_normal((3, bs, bs))     # multiplies the pad
            strips[:, -1, :, 2 * bs:] = rng.standard_normal((3, bs, bs))
            Y = orc.bdmv(strips, xpad)
            S64 = strips.astype(np.float64)
            S64[:, 0, :, :bs] = 0
            S64[:, -1, :, 2 * bs:] = 0
            Ad = assemble_bdsv_dense(S64)
            N = nbr * bs
            x = xpad[:, bs:bs + N].astype(np.float64)
            want = np.einsum("sij,sj->si", Ad, x)
            bound = 3 * bs * eps * np.einsum("sij,sj->si", np.abs(Ad), np.abs(x)) * 1.01
            assert np.all(np.abs(Y[:, bs:bs + N] - want) <= bound + 1e-300)


def pin_bdmv_inverts_bdsv(orc):
    """bdmv applied to the bdsv solution gives back b to the backward-error bound (the
    two routines read the same strips with the same layout)."""
    rng = _rng(49)
    nbr, bs = 8, 6
    strips, xpad = _random_bdsv(rng, 3, nbr, bs)
    _, X, info = orc.bdsv(strips, xpad)
    assert np.all(info == 0)
    Y = orc.bdmv(strips, X)
    N = nbr * bs
    b = xpad[:, bs:bs + N]
    Ad = assemble_bdsv_dense(strips)
    scale = np.abs(Ad).sum(axis=2).max(axis=1) * np.abs(X).max(axis=1) + np.abs(b).max(axis=1)
    assert np.all(np.abs(Y[:, bs:bs + N] - b).max(axis=1) <= 8 * N * eps_of(np.float64) * scale)


def pin_lu_nan_candidates(orc):
    """NaN in the pivot column, worked by hand under the search's strict "larger magnitude"
    test from the row in place (BLAS i_amax's comparison): a NaN below never displaces the
    current best; a NaN in the row in place is never displaced, becomes the pivot and
    makes the step singular (!(|p| >= floor)), with a reciprocal of 1.

    * [[1, 0], [NaN, 1]]: row 1 stays (NaN > 1 is false); the multiplier NaN * 1 turns the
      trailing entry into NaN, so step 2 is singular: ipiv = [1, 2], info = 2.
    * [[NaN, 0], [2, 1]]: the NaN in place stays (2 > NaN is false): info = 1, and with a
      reciprocal of 1 the multiplier is 2 exactly and the trailing entry 1 - 2 * 0 = 1.
    * [[1, 0, 0], [NaN, 1, 0], [2, 0, 1]]: the finite 2 wins step 1 over the NaN below
      (ipiv[0] = 3); the NaN row then sits in place at step 2: ipiv = [3, 2, 3], info = 2.
    Failed systems return X = 0; both storage orders and both precisions agree."""
    nan = np.nan
    for dt in (np.float64, np.float32):
        for layout in (ROW_MAJOR, COL_MAJOR):
            b2 = np.ones((1, 2, 1), dt)
            LU, X, ipiv, info, _ = _lu(orc, np.array([[[1, 0], [nan, 1]]], dt), b2, layout)
            assert list(ipiv[0]) == [1, 2] and info[0] == 2 and np.all(X == 0)
            assert LU[0, 0, 0] == 1 and LU[0, 0, 1] == 0 and np.isnan(LU[0, 1, 0])
            LU, X, ipiv, info, _ = _lu(orc, np.array([[[nan, 0], [2, 1]]], dt), b2, layout)
            assert list(ipiv[0]) == [1, 2] and info[0] == 1 and np.all(X == 0)
            assert np.isnan(LU[0, 0, 0]) and LU[0, 1, 0] == 2 and LU[0, 1, 1] == 1
            A3 = np.array([[[1, 0, 0], [nan, 1, 0], [2, 0, 1]]], dt)
            LU, X, ipiv, info, _ = _lu(orc, A3, np.ones((1, 3, 1), dt), layout)
            assert list(ipiv[0]) == [3, 2, 3] and info[0] == 2 and np.all(X == 0)
            assert list(LU[0, 0]) == [2, 0, 1] and LU[0, 2, 0] == dt(0.5)


LU_PINS = [pin_lu_3x3_hand_worked, pin_lu_2x2_closed_form, pin_lu_cramer_bruteforce,
           pin_lu_reconstruction, pin_lu_matches_lapack, pin_lu_info_contract,
           pin_lu_layout_invariance, pin_lu_near_tie_flag, pin_lu_nan_candidates]
CHOL_PINS = [pin_chol_hand_worked, pin_chol_2x2_closed_form,
             pin_chol_reconstruction_and_lapack, pin_chol_info_contract, pin_chol_upper_fill]
BDSV_PINS = [pin_bdsv_dense_equivalence, pin_bdsv_single_block_is_potrf,
             pin_bdsv_scalar_tridiagonal, pin_bdsv_info]
def pin_interleaved_literal(orc):
    """TDLS batched layouts, element e of system s at base_s[e * stride]: three 1x1
    systems in blocks of two (AoSoA, the last block ragged). A = (2, 4 | 0.5, pad),
    b = (1, 3 | 5, pad) as stored; x_s = b_s / a_s exactly: (0.5, 0.75 | 10), the pad
    untouched; Cholesky on a = (4, 16 | 0.25) gives l = (2, 4 | 0.5)."""
    nan = np.nan
    A = np.array([2.0, 4.0, 0.5, nan])
    B = np.array([1.0, 3.0, 5.0, nan])
    LU, X, ipiv, info, _ = orc.getrf_getrs_il(A, B, 1, 1, 3, 2, ROW_MAJOR)
    assert np.array_equal(X[:3], [0.5, 0.75, 10.0]) and np.isnan(X[3])
    assert np.array_equal(LU[:3], A[:3]) and np.isnan(LU[3])
    assert list(ipiv[:3]) == [1, 1, 1] and list(info) == [0, 0, 0]
    # two systems of order 2 in one block of two: element e of system s at 2e + s
    A2 = np.array([[[0.0, 1.0], [1.0, 0.0]], [[4.0, 2.0], [2.0, 2.0]]])
    B2 = np.array([[[3.0], [5.0]], [[2.0], [2.0]]])
    flatA = np.array([0.0, 4.0, 1.0, 2.0, 1.0, 2.0, 0.0, 2.0])
    flatB = np.array([3.0, 2.0, 5.0, 2.0])
    _, X2, p2, _, _ = orc.getrf_getrs_il(flatA, flatB, 2, 1, 2, 2, ROW_MAJOR)
    # system 0: the permutation [[0,1],[1,0]] swaps b; system 1: x = (0, 1) by Cramer
    assert np.array_equal(X2, [5.0, 0.0, 3.0, 1.0]) and list(p2) == [2, 1, 2, 2]
    assert np.array_equal(interleave(A2, 2), flatA) and np.array_equal(interleave(B2, 2), flatB)
    L, Xc, infc = orc.potrf_potrs_il(np.array([4.0, 16.0, 0.25, nan]),
                                     np.array([2.0, 8.0, 1.0, nan]), 1, 1, 3, 2)
    assert np.array_equal(L[:3], [2.0, 4.0, 0.5]) and np.isnan(L[3])
    assert np.array_equal(Xc[:3], [0.5, 0.5, 4.0]) and list(infc) == [0, 0, 0]


def pin_interleaved_layouts(orc):
    """The interleaved drivers equal the per-system ones on the same systems, bit for bit,
    for AoS (w = 1), AoSoA with a ragged last block, SoA (w = batch) and SoA with spare
    capacity (w > batch), both storage orders, LU and both Cholesky fills; the slots of
    the last block past the batch are never written."""
    rng = _rng(77)
    for dt in (np.float32, np.float64):
        for (n, nrhs, batch, w) in [(5, 2, 7, 1), (5, 2, 7, 3), (5, 2, 7, 7), (4, 1, 6, 16),
                                    (16, 4, 33, 32), (3, 3, 10, 4)]:
            for layout in (ROW_MAJOR, COL_MAJOR):
                Al = rng.standard_normal((batch, n, n)).astype(dt)
                Al[1, :, 0] = 0                     # a singular system
                A = to_storage(Al, layout)
                B = to_storage(rng.standard_normal((batch, n, nrhs)).astype(dt), layout)
                ref = orc.getrf_getrs(A, B, layout)
                got = orc.getrf_getrs_il(interleave(A, w), interleave(B, w), n, nrhs, batch, w,
                                         layout)
                assert np.array_equal(deinterleave(got[0], batch, w, A.shape[1:]), ref[0])
                assert np.array_equal(deinterleave(got[1], batch, w, B.shape[1:]), ref[1])
                assert np.array_equal(deinterleave(got[2], batch, w, (n,)), ref[2])
                assert np.array_equal(got[3], ref[3]) and np.array_equal(got[4], ref[4])
                pads = np.isnan(interleave(A, w))
                assert np.all(np.isnan(got[0][pads]))
                G = rng.standard_normal((batch, n, n)).astype(np.float64)
                Sl = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dt)
                Sl[2, n - 1, n - 1] = -1.0          # a failing minor
                for fill in (0, 1):
                    Sa = to_storage(Sl, layout)
                    r2 = orc.potrf_potrs(Sa, B, layout, fill=fill)
                    g2 = orc.potrf_potrs_il(interleave(Sa, w), interleave(B, w), n, nrhs, batch,
                                            w, layout, fill)
                    assert np.array_equal(deinterleave(g2[0], batch, w, Sa.shape[1:]), r2[0])
                    assert np.array_equal(deinterleave(g2[1], batch, w, B.shape[1:]), r2[1])
                    assert np.array_equal(g2[2], r2[2]) and g2[2][2] == n


def pin_interleaved_contract_options(orc):
    """The interleaved drivers with a pivot threshold or the RUDA status contract equal the
    per-system contract drivers on the same systems, bit for bit (ipiv -1 and zeros for a
    failed RUDA system included), the slots past the batch untouched."""
    rng = _rng(78)
    for dt in (np.float32, np.float64):
        for (n, nrhs, batch, w) in [(6, 2, 11, 4), (17, 3, 9, 9), (5, 1, 7, 16)]:
            for layout in (ROW_MAJOR, COL_MAJOR):
                Al = rng.standard_normal((batch, n, n)).astype(dt)
                Al[1, 0, 0] = np.inf                   # RUDA -1
                Al[2, :, 1] = 0                        # a singular system
                A = to_storage(Al, layout)
                B = to_storage(rng.standard_normal((batch, n, nrhs)).astype(dt), layout)
                for tau, ruda in ((0.5, 0), (1.0, 1), (0.3, 1)):
                    ref = orc.getrf_getrs_ex(A, B, layout, tau=tau, ruda=ruda)
                    got = orc.getrf_getrs_il(interleave(A, w), interleave(B, w), n, nrhs, batch,
                                             w, layout, tau=tau, ruda=ruda)
                    assert np.array_equal(deinterleave(got[0], batch, w, A.shape[1:]), ref[0],
                                          equal_nan=True)
                    assert np.array_equal(deinterleave(got[1], batch, w, B.shape[1:]), ref[1])
                    assert np.array_equal(deinterleave(got[2], batch, w, (n,)), ref[2])
                    assert np.array_equal(got[3], ref[3])
                    assert np.all(np.isnan(got[0][np.isnan(interleave(A, w))]))
                G = rng.standard_normal((batch, n, n))
                Sl = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dt)
                Sl[3, n - 1, 0] += 1.0                 # RUDA -2 (not symmetric)
                Sl[4, n // 2, n // 2] = -1.0           # a failing minor
                Sa = to_storage(Sl, layout)
                for fill in (0, 1):
                    r2 = orc.potrf_potrs_ex(Sa, B, layout, fill=fill, ruda=1)
                    g2 = orc.potrf_potrs_il(interleave(Sa, w), interleave(B, w), n, nrhs, batch,
                                            w, layout, fill, ruda=1)
                    assert np.array_equal(deinterleave(g2[0], batch, w, Sa.shape[1:]), r2[0])
                    assert np.array_equal(deinterleave(g2[1], batch, w, B.shape[1:]), r2[1])
                    assert np.array_equal(g2[2], r2[2]) and g2[2][3] == -2


def pin_ruda_scaling(orc):
    """RUDA's scaling by the largest magnitude of the matrix, with U's scale restored at the
    end (RUDA docs, unchanged numerical contract). Dividing by a power of two is exact and
    commutes with every rounding of the sweep, so with max |a_ij| a power of two the result
    is the unscaled one bit for bit; for any other maximum the factor reconstructs P A =
    L U and the solution meets the backward-error bound; a zero matrix is left unscaled
    (singular at step 1) and a non-finite input fails with -1 under the RUDA contract."""
    rng = _rng(91)
    for dt in (np.float32, np.float64):
        eps = eps_of(dt)
        for layout in (ROW_MAJOR, COL_MAJOR):
            for n, nrhs in ((1, 1), (5, 2), (16, 4), (33, 3)):
                Al = rng.uniform(-1, 1, (6, n, n)).astype(dt)
                Al[0, 0, n - 1] = 4.0               # max |a| = 4
                Al[1] *= dt(2.0 ** -5)
                Al[1, n - 1, 0] = -dt(2.0 ** -4)     # max |a| = 1/16
                Al[2, 0, 0] = -dt(2.0 ** 20)        # max |a| = 2^20
                Al[3] = 0
                Al[3, 0, 0] = 8.0
                A = to_storage(Al[:4], layout)
                B = to_storage(rng.standard_normal((4, n, nrhs)).astype(dt), layout)
                for tau, ruda in ((1.0, 0), (0.5, 1)):
                    r0 = orc.getrf_getrs_ex(A, B, layout, tau=tau, ruda=ruda)
                    r1 = orc.getrf_getrs_ex(A, B, layout, tau=tau, ruda=ruda, scale=1)
                    assert all(np.array_equal(x, y) for x, y in zip(r0, r1)), (n, tau)
                # a maximum that is not a power of two
                Ag = rng.uniform(-1, 1, (7, n, n)).astype(dt) * dt(3.7)
                Bg = rng.standard_normal((7, n, nrhs)).astype(dt)
                LU, X, ipiv, info, _ = orc.getrf_getrs_ex(to_storage(Ag, layout),
                                                          to_storage(Bg, layout), layout,
                                                          scale=1)
                LU, X = from_storage(LU, layout), from_storage(X, layout)
                ok = info == 0
                assert ok.sum() >= 5
                be = backward_error(Ag[ok].astype(np.float64), X[ok], Bg[ok])
                assert np.all(be <= 8 * n * eps)
                for sidx in np.nonzero(ok)[0]:
                    L, U = unpack_lu(LU[sidx])
                    PA = Ag[sidx].astype(np.float64)[lapack_perm(ipiv[sidx])]
                    nA = np.abs(Ag[sidx]).sum(axis=1).max()
                    assert np.abs(PA - L @ U).max() <= 4 * n * eps * nA
        Z = np.zeros((1, 3, 3), dt)
        r0 = orc.getrf_getrs_ex(Z, np.ones((1, 3, 1), dt), ROW_MAJOR)
        r1 = orc.getrf_getrs_ex(Z, np.ones((1, 3, 1), dt), ROW_MAJOR, scale=1)
        assert all(np.array_equal(x, y) for x, y in zip(r0, r1)) and r1[3][0] == 1
        Ai = np.eye(3, dtype=dt)[None].copy()
        Ai[0, 1, 2] = np.inf
        r = orc.getrf_getrs_ex(Ai, np.ones((1, 3, 1), dt), ROW_MAJOR, ruda=1, scale=1)
        assert r[3][0] == -1 and np.all(r[2] == -1)


def pin_mirror_scaling(orc):
    """The row-major reading (S = A^T, the stored row-major array read column-major) with
    RUDA's max-abs scaling: a maximum that is a power of two divides and multiplies back
    exactly, so the result is the unscaled reading's bit for bit; for any other maximum
    the stored factor reconstructs P S = L U with the restored U, and X solves A x = b to
    the backward-error bound; column-major storage (S = A) is the plain scaled call."""
    rng = _rng(93)
    for dt in (np.float32, np.float64):
        eps = eps_of(dt)
        for n, nrhs in ((1, 1), (5, 2), (16, 4), (33, 3)):
            Al = rng.uniform(-1, 1, (4, n, n)).astype(dt)
            Al[0, n - 1, 0] = 4.0
            Al[1] *= dt(2.0 ** -5)
            Al[1, 0, n - 1] = -dt(2.0 ** -4)
            Al[2, 0, 0] = -dt(2.0 ** 20)
            A = to_storage(Al[:3], ROW_MAJOR)
            B = rng.standard_normal((3, n, nrhs)).astype(dt)
            for tau in (1.0, 0.5):
                r0 = orc.getrf_getrs_mirror(A, B, ROW_MAJOR, tau=tau)
                r1 = orc.getrf_getrs_mirror(A, B, ROW_MAJOR, tau=tau, scale=1)
                assert all(np.array_equal(x, y) for x, y in zip(r0, r1)), (n, tau)
            Ag = rng.uniform(-1, 1, (6, n, n)).astype(dt) * dt(3.7)
            Bg = rng.standard_normal((6, n, nrhs)).astype(dt)
            F, X, ipiv, info, _ = orc.getrf_getrs_mirror(Ag, Bg, ROW_MAJOR, scale=1)
            ok = info == 0
            assert ok.sum() >= 4
            be = backward_error(Ag[ok].astype(np.float64), X[ok], Bg[ok])
            assert np.all(be <= 8 * n * eps), be
            for sidx in np.nonzero(ok)[0]:
                S = np.swapaxes(Ag[sidx], 0, 1).astype(np.float64)   # A^T
                L, U = unpack_lu(np.swapaxes(F[sidx], 0, 1))           # the factor of S
                nS = np.abs(S).sum(axis=1).max()
                assert np.abs(S[lapack_perm(ipiv[sidx])] - L @ U).max() <= 4 * n * eps * nS
            Ac = to_storage(Ag, COL_MAJOR)
            Bc = to_storage(Bg, COL_MAJOR)
            rc = orc.getrf_getrs_mirror(Ac, Bc, COL_MAJOR, scale=1)
            rd = orc.getrf_getrs_ex(Ac, Bc, COL_MAJOR, scale=1)
            assert all(np.array_equal(x, y) for x, y in zip(rc, rd))
        # worked by hand: A = s I with s subnormal. Unscaled, the first pivot is below the
        # smallest normal: info = 1, X = 0. Scaled, the sweep sees I (info = 0), U = s I is
        # restored, and its subnormal diagonal takes the reciprocal 1: z = b, w = z, x = b.
        sub = np.finfo(dt).smallest_subnormal * 8
        As = np.array([[[sub, 0.0], [0.0, sub]]], dt)
        Bs = np.array([[[3.0], [-5.0]]], dt)
        _, X0, _, info0, _ = orc.getrf_getrs_mirror(As, Bs, ROW_MAJOR)
        assert info0[0] == 1 and np.all(X0 == 0)
        _, X1, ip1, info1, _ = orc.getrf_getrs_mirror(As, Bs, ROW_MAJOR, scale=1)
        assert info1[0] == 0 and np.array_equal(X1, Bs) and list(ip1[0]) == [1, 2]


def pin_interleaved_split_and_mirror(orc):
    """TDLS batched layouts on the separate factor and solve steps and on the row-major
    reading. Literal 1x1 systems in blocks of two (the last block ragged): getrf leaves
    a = (2, 4 | 0.5) with ipiv 1, getrs gives x = b / a = (0.5, 0.75 | 10); potrf gives
    l = (2, 4 | 0.5) for a = (4, 16 | 0.25), potrs x = b (1/l)(1/l) = (0.5, 0.5 | 4); the
    pads never written. Then random systems: every interleaved driver equals its
    per-system driver on the same systems bit for bit (AoS, ragged AoSoA, SoA, SoA with
    spare capacity, both storage orders, both fills, a threshold and the scaling for the
    row-major reading), and getrf then getrs equals the fused interleaved call."""
    nan = np.nan
    F, p, info, _ = orc.getrf_il(np.array([2.0, 4.0, 0.5, nan]), 1, 3, 2)
    assert np.array_equal(F[:3], [2.0, 4.0, 0.5]) and np.isnan(F[3])
    assert list(p[:3]) == [1, 1, 1] and list(info) == [0, 0, 0]
    X = orc.getrs_il(F, p, np.array([1.0, 3.0, 5.0, nan]), 1, 1, 3, 2)
    assert np.array_equal(X[:3], [0.5, 0.75, 10.0]) and np.isnan(X[3])
    L, infc = orc.potrf_il(np.array([4.0, 16.0, 0.25, nan]), 1, 3, 2)
    assert np.array_equal(L[:3], [2.0, 4.0, 0.5]) and np.isnan(L[3]) and list(infc) == [0] * 3
    Xc = orc.potrs_il(L, np.array([2.0, 8.0, 1.0, nan]), 1, 1, 3, 2)
    assert np.array_equal(Xc[:3], [0.5, 0.5, 4.0]) and np.isnan(Xc[3])
    rng = _rng(94)
    for dt in (np.float32, np.float64):
        for (n, nrhs, batch, w) in [(5, 2, 7, 1), (5, 2, 7, 3), (5, 2, 7, 7), (4, 1, 6, 16),
                                    (16, 4, 33, 32), (33, 2, 5, 2)]:
            for layout in (ROW_MAJOR, COL_MAJOR):
                Al = rng.standard_normal((batch, n, n)).astype(dt)
                Al[1, :, 0] = 0
                A = to_storage(Al, layout)
                B = to_storage(rng.standard_normal((batch, n, nrhs)).astype(dt), layout)
                di = lambda f, shape: deinterleave(f, batch, w, shape)   # noqa: E731
                LUo, ipo, info_o, tie_o = orc.getrf(A, layout)
                LUi, ipi, infi, tiei = orc.getrf_il(interleave(A, w), n, batch, w, layout)
                assert np.array_equal(di(LUi, A.shape[1:]), LUo)
                assert np.array_equal(di(ipi, (n,)), ipo) and np.array_equal(infi, info_o)
                assert np.array_equal(tiei, tie_o)
                assert np.all(np.isnan(LUi[np.isnan(interleave(A, w))]))
                Xo = orc.getrs(LUo, ipo, B, layout)
                Xi = orc.getrs_il(LUi, ipi, interleave(B, w), n, nrhs, batch, w, layout)
                assert np.array_equal(di(Xi, B.shape[1:]), Xo)
                fused = orc.getrf_getrs_il(interleave(A, w), interleave(B, w), n, nrhs, batch,
                                           w, layout)
                ok = info_o == 0
                assert np.array_equal(di(fused[1], B.shape[1:])[ok], Xo[ok])
                for tau, scale in ((1.0, 0), (0.5, 0), (1.0, 1)):
                    mo = orc.getrf_getrs_mirror(A, B, layout, tau=tau, scale=scale)
                    mi = orc.getrf_getrs_mirror_il(interleave(A, w), interleave(B, w), n, nrhs,
                                                   batch, w, layout, tau=tau, scale=scale)
                    assert np.array_equal(di(mi[0], A.shape[1:]), mo[0])
                    assert np.array_equal(di(mi[1], B.shape[1:]), mo[1])
                    assert np.array_equal(di(mi[2], (n,)), mo[2])
                    assert np.array_equal(mi[3], mo[3]) and np.array_equal(mi[4], mo[4])
                G = rng.standard_normal((batch, n, n))
                Sl = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dt)
                Sl[2 % batch, n - 1, n - 1] = -1.0
                for fill in (0, 1):
                    Sa = to_storage(Sl, layout)
                    Lo, io = orc.potrf(Sa, layout, fill=fill)
                    Li, ii = orc.potrf_il(interleave(Sa, w), n, batch, w, layout, fill)
                    assert np.array_equal(di(Li, Sa.shape[1:]), Lo) and np.array_equal(ii, io)
                    Xo = orc.potrs(Lo, B, layout, fill=fill)
                    Xi = orc.potrs_il(Li, interleave(B, w), n, nrhs, batch, w, layout, fill)
                    assert np.array_equal(di(Xi, B.shape[1:]), Xo)


SPLIT_PINS = [pin_getrs_composition, pin_getrs_permutation_only, pin_getrs_cramer,
              pin_potrs_composition, pin_potrs_diagonal, pin_potrs_dense, pin_bdsv_split]
BDMV_PINS = [pin_bdmv_exact_integers, pin_bdmv_dense, pin_bdmv_inverts_bdsv]
VARIANT_PINS = [pin_threshold_pivoting, pin_ruda_status_lu, pin_ruda_status_chol,
                pin_tdls_row_major_reading, pin_ruda_scaling, pin_mirror_scaling]
LAYOUT_PINS = [pin_interleaved_literal, pin_interleaved_layouts,
               pin_interleaved_contract_options, pin_interleaved_split_and_mirror]
ALL_PINS = (LU_PINS + CHOL_PINS + BDSV_PINS + SPLIT_PINS + BDMV_PINS + VARIANT_PINS +
            LAYOUT_PINS)


def failing_pins(orc, pins=ALL_PINS):
    """Names of the pins that fail (or raise) on this oracle."""
    bad = []
    for p in pins:
        try:
            p(orc)
        except Exception:  # noqa: BLE001 - any failure counts as a tripped pin
            bad.append(p.__name__)
    return bad
