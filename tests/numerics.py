"""Error measures used by the pins and the parity tests (NumPy, test-only).

The residual b - A x is accumulated in double-double arithmetic (Dekker's splitting for
exact products and Knuth's TwoSum for exact sums, as in Ogita, Rump and Oishi,
"Accurate sum and dot product", SIAM J. Sci. Comput. 2005), so that the checker's own
rounding stays far below the FP64 backward-error bound it checks.
"""
from __future__ import annotations

import numpy as np

_SPLIT = 134217729.0  # 2**27 + 1


def _two_sum(a, b):
    s = a + b
    bb = s - a
    e = (a - (s - bb)) + (b - bb)
    return s, e


def _split(a):
    c = _SPLIT * a
    hi = c - (c - a)
    return hi, a - hi


def _two_prod(a, b):
    p = a * b
    ah, al = _split(a)
    bh, bl = _split(b)
    e = ((ah * bh - p) + ah * bl + al * bh) + al * bl
    return p, e


def residual_dd(A: np.ndarray, X: np.ndarray, B: np.ndarray) -> np.ndarray:
    """R = B - A X for logical (batch, n, n), (batch, n, k), (batch, n, k) arrays,
    accumulated in double-double and rounded to float64 at the end."""
    A = np.asarray(A, np.float64)
    X = np.asarray(X, np.float64)
    s = np.array(B, np.float64, copy=True)
    c = np.zeros_like(s)
    n = A.shape[-1]
    for j in range(n):
        p, e = _two_prod(-A[:, :, j:j + 1], X[:, j:j + 1, :])
        s, e2 = _two_sum(s, p)
        c = c + (e + e2)
    return s + c


def inf_norm_rows(A: np.ndarray) -> np.ndarray:
    """Matrix infinity norm per system (max row sum)."""
    return np.abs(np.asarray(A, np.float64)).sum(axis=-1).max(axis=-1)


def backward_error(A: np.ndarray, X: np.ndarray, B: np.ndarray) -> np.ndarray:
    """Per system and right-hand side column j:
    ||A x_j - b_j||_inf / (||A||_inf ||x_j||_inf + ||b_j||_inf); returns the max over j."""
    R = residual_dd(A, X, B)
    rn = np.abs(R).max(axis=1)                       # (batch, k)
    an = inf_norm_rows(A)[:, None]
    xn = np.abs(np.asarray(X, np.float64)).max(axis=1)
    bn = np.abs(np.asarray(B, np.float64)).max(axis=1)
    den = an * xn + bn
    with np.errstate(invalid="ignore", divide="ignore"):
        be = np.where(den > 0, rn / den, np.where(rn > 0, np.inf, 0.0))
    return be.max(axis=1)


def forward_error(X: np.ndarray, Xref: np.ndarray) -> np.ndarray:
    """||x - x_ref||_inf / ||x_ref||_inf per system (all right-hand sides together)."""
    X = np.asarray(X, np.float64).reshape(X.shape[0], -1)
    Xr = np.asarray(Xref, np.float64).reshape(Xref.shape[0], -1)
    num = np.abs(X - Xr).max(axis=1)
    den = np.abs(Xr).max(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        return np.where(den > 0, num / den, num)


def eps_of(dtype) -> float:
    return float(np.finfo(dtype).eps)


def lapack_perm(ipiv: np.ndarray) -> np.ndarray:
    """Row order produced by applying the 1-based swap sequence ipiv to 0..n-1."""
    n = ipiv.shape[-1]
    perm = np.arange(n)
    for k in range(n):
        p = int(ipiv[k]) - 1
        perm[k], perm[p] = perm[p], perm[k]
    return perm


def unpack_lu(LU: np.ndarray):
    """Logical LU (n x n) -> (unit lower L, upper U) as float64."""
    LU = np.asarray(LU, np.float64)
    n = LU.shape[-1]
    L = np.tril(LU, -1) + np.eye(n)
    U = np.triu(LU)
    return L, U
