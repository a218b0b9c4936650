"""Sequential CPU oracle for the batched small dense solvers (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline / reference arm
of ``bench.py`` may import this package. The CUDA library never links, loads or calls
it, and it imports nothing from the CUDA side.

The arithmetic lives in ``oracle.cpp`` (plain sequential C++, one system at a time, in
the dtype of the inputs). This module only builds that file with g++ and marshals
NumPy arrays: every function copies its inputs and returns new arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_default = None

ROW_MAJOR = 0
COL_MAJOR = 1
LOWER = 0
UPPER = 1


def compile_library(src: str, out: str) -> str:
    """g++ -O2 without FMA contraction or fast-math; writes ``out`` atomically."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", "-o", tmp, src]
    subprocess.check_call(cmd)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.cpp into _build/liboracle.so if it is missing or stale."""
    stale = (not os.path.exists(_SO)) or os.path.getmtime(_SO) < os.path.getmtime(_SRC)
    if force or stale:
        compile_library(_SRC, _SO)
    return _SO


class Oracle:
    """ctypes view of one compiled oracle library (the default one, or a variant)."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        for name in ("oracle_getrf_getrs_f32", "oracle_getrf_getrs_f64"):
            getattr(lib, name).argtypes = [i32, i32, i32, i64, vp, vp, vp, vp, vp, i32]
            getattr(lib, name).restype = i32
        for name in ("oracle_potrf_potrs_f32", "oracle_potrf_potrs_f64"):
            getattr(lib, name).argtypes = [i32, i32, i32, i32, i64, vp, vp, vp, i32]
            getattr(lib, name).restype = i32
        for name in ("oracle_bdsv_f32", "oracle_bdsv_f64"):
            getattr(lib, name).argtypes = [i32, i32, i64, vp, vp, vp, i32]
            getattr(lib, name).restype = i32
        sig = {
            "getrf": [i32, i32, i64, vp, vp, vp, vp, i32],
            "getrs": [i32, i32, i32, i64, vp, vp, vp, i32],
            "potrf": [i32, i32, i32, i64, vp, vp, i32],
            "potrs": [i32, i32, i32, i32, i64, vp, vp, i32],
            "bdsv_factor": [i32, i32, i64, vp, vp, i32],
            "bdsv_solve": [i32, i32, i64, vp, vp, i32],
            "bdmv": [i32, i32, i64, vp, vp, vp, i32],
        }
        sig["getrf_getrs_ex"] = [i32, i32, i32, i64, vp, vp, vp, vp, vp, ctypes.c_double, i32, i32,
                                 i32]
        sig["potrf_potrs_ex"] = [i32, i32, i32, i32, i64, vp, vp, vp, i32, i32]
        sig["getrf_getrs_mirror"] = [i32, i32, i32, i64, vp, vp, vp, vp, vp, ctypes.c_double, i32]
        sig["getrf_getrs_il"] = [i32, i32, i32, i64, i64, vp, vp, vp, vp, vp, ctypes.c_double,
                                 i32, i32, i32]
        sig["potrf_potrs_il"] = [i32, i32, i32, i32, i64, i64, vp, vp, vp, i32, i32]
        sig["getrf_getrs_mirror_ex"] = [i32, i32, i32, i64, i64, vp, vp, vp, vp, vp,
                                        ctypes.c_double, i32, i32]
        sig["getrf_il"] = [i32, i32, i64, i64, vp, vp, vp, vp, i32]
        sig["getrs_il"] = [i32, i32, i32, i64, i64, vp, vp, vp, i32]
        sig["potrf_il"] = [i32, i32, i32, i64, i64, vp, vp, i32]
        sig["potrs_il"] = [i32, i32, i32, i32, i64, i64, vp, vp, i32]
        for op, args in sig.items():
            for sfx in ("f32", "f64"):
                fn = getattr(lib, f"oracle_{op}_{sfx}")
                fn.argtypes = args
                fn.restype = i32
        self.lib = lib

    def getrf_getrs(self, A, B, layout: int = ROW_MAJOR, nthreads: int = 1):
        """LU with partial pivoting + solve, one system at a time.

        A: (batch, n, n) and B: raw storage in ``layout`` order (see gen.workloads).
        Returns (LU, X, ipiv, info, tie_step) with LU/X in the inputs' storage order.
        """
        A = np.ascontiguousarray(A).copy()
        B = np.ascontiguousarray(B, dtype=A.dtype).copy()
        batch, n = A.shape[0], A.shape[1]
        nrhs = B.shape[-1] if layout == ROW_MAJOR else B.shape[-2]
        ipiv = np.zeros((batch, n), np.int32)
        info = np.zeros(batch, np.int32)
        tie = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_getrf_getrs_" + _suffix(A.dtype))
        rc = fn(layout, n, nrhs, batch, _ptr(A), _ptr(B), _ptr(ipiv), _ptr(info), _ptr(tie),
                nthreads)
        if rc != 0:
            raise ValueError("oracle getrf_getrs rejected its arguments")
        return A, B, ipiv, info, tie

    def potrf_potrs(self, A, B, layout: int = COL_MAJOR, nthreads: int = 1, fill: int = LOWER):
        """Cholesky + solve, one system at a time (fill LOWER: A = L L^T in the lower
        triangle; UPPER: A = U^T U in the upper one). Returns (factor, X, info)."""
        A = np.ascontiguousarray(A).copy()
        B = np.ascontiguousarray(B, dtype=A.dtype).copy()
        batch, n = A.shape[0], A.shape[1]
        nrhs = B.shape[-1] if layout == ROW_MAJOR else B.shape[-2]
        info = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_potrf_potrs_" + _suffix(A.dtype))
        rc = fn(layout, fill, n, nrhs, batch, _ptr(A), _ptr(B), _ptr(info), nthreads)
        if rc != 0:
            raise ValueError("oracle potrf_potrs rejected its arguments")
        return A, B, info

    def bdsv(self, strips, xpad, nthreads: int = 1):
        """Block-tridiagonal block-Cholesky solve.

        strips: (batch, nbr, bs, 3*bs) [L|D|R]; xpad: (batch, (nbr+2)*bs).
        Returns (factored strips, padded solution, info).
        """
        S = np.ascontiguousarray(strips).copy()
        X = np.ascontiguousarray(xpad, dtype=S.dtype).copy()
        batch, nbr, bs = S.shape[0], S.shape[1], S.shape[2]
        info = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_bdsv_" + _suffix(S.dtype))
        rc = fn(nbr, bs, batch, _ptr(S), _ptr(X), _ptr(info), nthreads)
        if rc != 0:
            raise ValueError("oracle bdsv rejected its arguments")
        return S, X, info

    # --- factor once, solve per right-hand side -------------------------------------
    def getrf(self, A, layout: int = ROW_MAJOR, nthreads: int = 1):
        """LU with partial pivoting only. Returns (LU, ipiv, info, tie_step)."""
        A = np.ascontiguousarray(A).copy()
        batch, n = A.shape[0], A.shape[1]
        ipiv = np.zeros((batch, n), np.int32)
        info = np.zeros(batch, np.int32)
        tie = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_getrf_" + _suffix(A.dtype))
        if fn(layout, n, batch, _ptr(A), _ptr(ipiv), _ptr(info), _ptr(tie), nthreads) != 0:
            raise ValueError("oracle getrf rejected its arguments")
        return A, ipiv, info, tie

    def getrs(self, LU, ipiv, B, layout: int = ROW_MAJOR, nthreads: int = 1):
        """Solve with a stored LU factor and swap sequence. Returns X."""
        LU = np.ascontiguousarray(LU)
        ipiv = np.ascontiguousarray(ipiv, dtype=np.int32)
        B = np.ascontiguousarray(B, dtype=LU.dtype).copy()
        batch, n = LU.shape[0], LU.shape[1]
        nrhs = B.shape[-1] if layout == ROW_MAJOR else B.shape[-2]
        fn = getattr(self.lib, "oracle_getrs_" + _suffix(LU.dtype))
        if fn(layout, n, nrhs, batch, _ptr(LU), _ptr(ipiv), _ptr(B), nthreads) != 0:
            raise ValueError("oracle getrs rejected its arguments")
        return B

    def potrf(self, A, layout: int = COL_MAJOR, nthreads: int = 1, fill: int = LOWER):
        """Cholesky only (fill as potrf_potrs). Returns (factor, info)."""
        A = np.ascontiguousarray(A).copy()
        batch, n = A.shape[0], A.shape[1]
        info = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_potrf_" + _suffix(A.dtype))
        if fn(layout, fill, n, batch, _ptr(A), _ptr(info), nthreads) != 0:
            raise ValueError("oracle potrf rejected its arguments")
        return A, info

    def potrs(self, L, B, layout: int = COL_MAJOR, nthreads: int = 1, fill: int = LOWER):
        """Solve with a stored Cholesky factor (fill as potrf_potrs). Returns X."""
        L = np.ascontiguousarray(L)
        B = np.ascontiguousarray(B, dtype=L.dtype).copy()
        batch, n = L.shape[0], L.shape[1]
        nrhs = B.shape[-1] if layout == ROW_MAJOR else B.shape[-2]
        fn = getattr(self.lib, "oracle_potrs_" + _suffix(L.dtype))
        if fn(layout, fill, n, nrhs, batch, _ptr(L), _ptr(B), nthreads) != 0:
            raise ValueError("oracle potrs rejected its arguments")
        return B

    def bdsv_factor(self, strips, nthreads: int = 1):
        """Block-Cholesky factor sweep in place. Returns (factored strips, info)."""
        S = np.ascontiguousarray(strips).copy()
        batch, nbr, bs = S.shape[0], S.shape[1], S.shape[2]
        info = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_bdsv_factor_" + _suffix(S.dtype))
        if fn(nbr, bs, batch, _ptr(S), _ptr(info), nthreads) != 0:
            raise ValueError("oracle bdsv_factor rejected its arguments")
        return S, info

    def bdsv_solve(self, strips, xpad, nthreads: int = 1):
        """Forward/backward block substitution with factored strips. Returns the padded x."""
        S = np.ascontiguousarray(strips)
        X = np.ascontiguousarray(xpad, dtype=S.dtype).copy()
        batch, nbr, bs = S.shape[0], S.shape[1], S.shape[2]
        fn = getattr(self.lib, "oracle_bdsv_solve_" + _suffix(S.dtype))
        if fn(nbr, bs, batch, _ptr(S), _ptr(X), nthreads) != 0:
            raise ValueError("oracle bdsv_solve rejected its arguments")
        return X

    def bdmv(self, strips, xpad, ypad=None, nthreads: int = 1):
        """Block-tridiagonal matvec y = A x on padded vectors (y's pads kept from ypad, or
        zero). Returns the padded y."""
        S = np.ascontiguousarray(strips)
        X = np.ascontiguousarray(xpad, dtype=S.dtype)
        Y = (np.zeros_like(X) if ypad is None
             else np.ascontiguousarray(ypad, dtype=S.dtype).copy())
        batch, nbr, bs = S.shape[0], S.shape[1], S.shape[2]
        fn = getattr(self.lib, "oracle_bdmv_" + _suffix(S.dtype))
        if fn(nbr, bs, batch, _ptr(S), _ptr(X), _ptr(Y), nthreads) != 0:
            raise ValueError("oracle bdmv rejected its arguments")
        return Y

    # --- contract variants ------------------------------------------------------------
    def getrf_getrs_ex(self, A, B, layout: int = ROW_MAJOR, tau: float = 1.0, ruda: int = 0,
                       nthreads: int = 1, scale: int = 0):
        """LU + solve with TDLS threshold pivoting (tau), the RUDA status contract and/or
        RUDA's scaling by the largest magnitude of the matrix (scale). Returns (LU, X,
        ipiv, info, tie_step)."""
        A = np.ascontiguousarray(A).copy()
        B = np.ascontiguousarray(B, dtype=A.dtype).copy()
        batch, n = A.shape[0], A.shape[1]
        nrhs = B.shape[-1] if layout == ROW_MAJOR else B.shape[-2]
        ipiv = np.zeros((batch, n), np.int32)
        info = np.zeros(batch, np.int32)
        tie = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_getrf_getrs_ex_" + _suffix(A.dtype))
        if fn(layout, n, nrhs, batch, _ptr(A), _ptr(B), _ptr(ipiv), _ptr(info), _ptr(tie),
              float(tau), int(ruda), int(scale), nthreads) != 0:
            raise ValueError("oracle getrf_getrs_ex rejected its arguments")
        return A, B, ipiv, info, tie

    def potrf_potrs_ex(self, A, B, layout: int = COL_MAJOR, fill: int = LOWER, ruda: int = 0,
                       nthreads: int = 1):
        """Cholesky + solve under the RUDA status contract. Returns (factor, X, info)."""
        A = np.ascontiguousarray(A).copy()
        B = np.ascontiguousarray(B, dtype=A.dtype).copy()
        batch, n = A.shape[0], A.shape[1]
        nrhs = B.shape[-1] if layout == ROW_MAJOR else B.shape[-2]
        info = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_potrf_potrs_ex_" + _suffix(A.dtype))
        if fn(layout, fill, n, nrhs, batch, _ptr(A), _ptr(B), _ptr(info), int(ruda), nthreads) != 0:
            raise ValueError("oracle potrf_potrs_ex rejected its arguments")
        return A, B, info

    def getrf_getrs_mirror(self, A, B, layout: int = ROW_MAJOR, tau: float = 1.0,
                           nthreads: int = 1, scale: int = 0):
        """TDLS row-major reading: factor S (the stored array read column-major, S = A^T for
        row-major storage), then U^T z = b, L^T w = z, x = P^T w; scale: RUDA's max-abs
        scaling of the factorization. Returns (S factored in the stored array, X, ipiv,
        info, tie_step)."""
        A = np.ascontiguousarray(A).copy()
        B = np.ascontiguousarray(B, dtype=A.dtype).copy()
        batch, n = A.shape[0], A.shape[1]
        nrhs = B.shape[-1] if layout == ROW_MAJOR else B.shape[-2]
        ipiv = np.zeros((batch, n), np.int32)
        info = np.zeros(batch, np.int32)
        tie = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_getrf_getrs_mirror_ex_" + _suffix(A.dtype))
        if fn(layout, n, nrhs, batch, 1, _ptr(A), _ptr(B), _ptr(ipiv), _ptr(info), _ptr(tie),
              float(tau), int(scale), nthreads) != 0:
            raise ValueError("oracle getrf_getrs_mirror rejected its arguments")
        return A, B, ipiv, info, tie


    def getrf_getrs_il(self, A, B, n: int, nrhs: int, batch: int, w: int,
                       layout: int = ROW_MAJOR, nthreads: int = 1, tau: float = 1.0,
                       ruda: int = 0, scale: int = 0):
        """LU + solve on interleaved batched storage (TDLS: element e of system s at
        base_s[e * w], base_s = (s // w) * w * size + s % w; w = 1 AoS, w >= batch SoA).
        A, B: flat arrays of ceil(batch / w) * w systems. Returns (A, B, ipiv, info,
        tie_step), ipiv flat and interleaved like A. tau and ruda: the contract options of
        getrf_getrs_ex."""
        A = np.ascontiguousarray(A).reshape(-1).copy()
        B = np.ascontiguousarray(B, dtype=A.dtype).reshape(-1).copy()
        nb = -(-batch // w) if batch else 0
        if A.size < nb * w * n * n or B.size < nb * w * n * nrhs:
            raise ValueError("interleaved buffers too small")
        ipiv = np.zeros(max(nb * w * n, 1), np.int32)
        info = np.zeros(batch, np.int32)
        tie = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_getrf_getrs_il_" + _suffix(A.dtype))
        if fn(layout, n, nrhs, batch, w, _ptr(A), _ptr(B), _ptr(ipiv), _ptr(info), _ptr(tie),
              float(tau), int(ruda), int(scale), nthreads) != 0:
            raise ValueError("oracle getrf_getrs_il rejected its arguments")
        return A, B, ipiv, info, tie

    def getrf_getrs_mirror_il(self, A, B, n: int, nrhs: int, batch: int, w: int,
                              layout: int = ROW_MAJOR, tau: float = 1.0, scale: int = 0,
                              nthreads: int = 1):
        """The row-major reading (getrf_getrs_mirror) on interleaved batched storage (see
        getrf_getrs_il). Returns (A, B, ipiv, info, tie_step), ipiv flat and interleaved."""
        A = np.ascontiguousarray(A).reshape(-1).copy()
        B = np.ascontiguousarray(B, dtype=A.dtype).reshape(-1).copy()
        nb = -(-batch // w) if batch else 0
        if A.size < nb * w * n * n or B.size < nb * w * n * nrhs:
            raise ValueError("interleaved buffers too small")
        ipiv = np.zeros(max(nb * w * n, 1), np.int32)
        info = np.zeros(batch, np.int32)
        tie = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_getrf_getrs_mirror_ex_" + _suffix(A.dtype))
        if fn(layout, n, nrhs, batch, w, _ptr(A), _ptr(B), _ptr(ipiv), _ptr(info), _ptr(tie),
              float(tau), int(scale), nthreads) != 0:
            raise ValueError("oracle getrf_getrs_mirror rejected its arguments")
        return A, B, ipiv, info, tie

    def getrf_il(self, A, n: int, batch: int, w: int, layout: int = ROW_MAJOR,
                 nthreads: int = 1):
        """getrf on interleaved storage. Returns (A, ipiv, info, tie_step)."""
        A = np.ascontiguousarray(A).reshape(-1).copy()
        nb = -(-batch // w) if batch else 0
        if A.size < nb * w * n * n:
            raise ValueError("interleaved buffers too small")
        ipiv = np.zeros(max(nb * w * n, 1), np.int32)
        info = np.zeros(batch, np.int32)
        tie = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_getrf_il_" + _suffix(A.dtype))
        if fn(layout, n, batch, w, _ptr(A), _ptr(ipiv), _ptr(info), _ptr(tie), nthreads) != 0:
            raise ValueError("oracle getrf_il rejected its arguments")
        return A, ipiv, info, tie

    def getrs_il(self, LU, ipiv, B, n: int, nrhs: int, batch: int, w: int,
                 layout: int = ROW_MAJOR, nthreads: int = 1):
        """getrs on interleaved storage (LU and ipiv as getrf_il leaves them). Returns B."""
        LU = np.ascontiguousarray(LU).reshape(-1)
        ipiv = np.ascontiguousarray(ipiv, dtype=np.int32).reshape(-1)
        B = np.ascontiguousarray(B, dtype=LU.dtype).reshape(-1).copy()
        fn = getattr(self.lib, "oracle_getrs_il_" + _suffix(LU.dtype))
        if fn(layout, n, nrhs, batch, w, _ptr(LU), _ptr(ipiv), _ptr(B), nthreads) != 0:
            raise ValueError("oracle getrs_il rejected its arguments")
        return B

    def potrf_il(self, A, n: int, batch: int, w: int, layout: int = COL_MAJOR,
                 fill: int = LOWER, nthreads: int = 1):
        """potrf on interleaved storage. Returns (A, info)."""
        A = np.ascontiguousarray(A).reshape(-1).copy()
        info = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_potrf_il_" + _suffix(A.dtype))
        if fn(layout, fill, n, batch, w, _ptr(A), _ptr(info), nthreads) != 0:
            raise ValueError("oracle potrf_il rejected its arguments")
        return A, info

    def potrs_il(self, L, B, n: int, nrhs: int, batch: int, w: int, layout: int = COL_MAJOR,
                 fill: int = LOWER, nthreads: int = 1):
        """potrs on interleaved storage. Returns B."""
        L = np.ascontiguousarray(L).reshape(-1)
        B = np.ascontiguousarray(B, dtype=L.dtype).reshape(-1).copy()
        fn = getattr(self.lib, "oracle_potrs_il_" + _suffix(L.dtype))
        if fn(layout, fill, n, nrhs, batch, w, _ptr(L), _ptr(B), nthreads) != 0:
            raise ValueError("oracle potrs_il rejected its arguments")
        return B

    def potrf_potrs_il(self, A, B, n: int, nrhs: int, batch: int, w: int,
                       layout: int = COL_MAJOR, fill: int = LOWER, nthreads: int = 1,
                       ruda: int = 0):
        """Cholesky + solve on interleaved batched storage (see getrf_getrs_il; ruda: the
        status contract of potrf_potrs_ex). Returns (A, B, info)."""
        A = np.ascontiguousarray(A).reshape(-1).copy()
        B = np.ascontiguousarray(B, dtype=A.dtype).reshape(-1).copy()
        nb = -(-batch // w) if batch else 0
        if A.size < nb * w * n * n or B.size < nb * w * n * nrhs:
            raise ValueError("interleaved buffers too small")
        info = np.zeros(batch, np.int32)
        fn = getattr(self.lib, "oracle_potrf_potrs_il_" + _suffix(A.dtype))
        if fn(layout, fill, n, nrhs, batch, w, _ptr(A), _ptr(B), _ptr(info), int(ruda),
              nthreads) != 0:
            raise ValueError("oracle potrf_potrs_il rejected its arguments")
        return A, B, info


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def getrf_getrs(A, B, layout: int = ROW_MAJOR, nthreads: int = 1):
    return default().getrf_getrs(A, B, layout, nthreads)


def potrf_potrs(A, B, layout: int = COL_MAJOR, nthreads: int = 1, fill: int = LOWER):
    return default().potrf_potrs(A, B, layout, nthreads, fill)


def bdsv(strips, xpad, nthreads: int = 1):
    return default().bdsv(strips, xpad, nthreads)


def getrf(A, layout: int = ROW_MAJOR, nthreads: int = 1):
    return default().getrf(A, layout, nthreads)


def getrs(LU, ipiv, B, layout: int = ROW_MAJOR, nthreads: int = 1):
    return default().getrs(LU, ipiv, B, layout, nthreads)


def potrf(A, layout: int = COL_MAJOR, nthreads: int = 1, fill: int = LOWER):
    return default().potrf(A, layout, nthreads, fill)


def potrs(L, B, layout: int = COL_MAJOR, nthreads: int = 1, fill: int = LOWER):
    return default().potrs(L, B, layout, nthreads, fill)


def bdsv_factor(strips, nthreads: int = 1):
    return default().bdsv_factor(strips, nthreads)


def bdsv_solve(strips, xpad, nthreads: int = 1):
    return default().bdsv_solve(strips, xpad, nthreads)


def bdmv(strips, xpad, ypad=None, nthreads: int = 1):
    return default().bdmv(strips, xpad, ypad, nthreads)


def getrf_getrs_ex(A, B, layout: int = ROW_MAJOR, tau: float = 1.0, ruda: int = 0,
                   nthreads: int = 1, scale: int = 0):
    return default().getrf_getrs_ex(A, B, layout, tau, ruda, nthreads, scale)


def potrf_potrs_ex(A, B, layout: int = COL_MAJOR, fill: int = LOWER, ruda: int = 0,
                   nthreads: int = 1):
    return default().potrf_potrs_ex(A, B, layout, fill, ruda, nthreads)


def getrf_getrs_mirror(A, B, layout: int = ROW_MAJOR, tau: float = 1.0, nthreads: int = 1,
                       scale: int = 0):
    return default().getrf_getrs_mirror(A, B, layout, tau, nthreads, scale)


def getrf_getrs_mirror_il(A, B, n, nrhs, batch, w, layout: int = ROW_MAJOR, tau: float = 1.0,
                          scale: int = 0, nthreads: int = 1):
    return default().getrf_getrs_mirror_il(A, B, n, nrhs, batch, w, layout, tau, scale, nthreads)


def getrf_il(A, n, batch, w, layout: int = ROW_MAJOR, nthreads: int = 1):
    return default().getrf_il(A, n, batch, w, layout, nthreads)


def getrs_il(LU, ipiv, B, n, nrhs, batch, w, layout: int = ROW_MAJOR, nthreads: int = 1):
    return default().getrs_il(LU, ipiv, B, n, nrhs, batch, w, layout, nthreads)


def potrf_il(A, n, batch, w, layout: int = COL_MAJOR, fill: int = LOWER, nthreads: int = 1):
    return default().potrf_il(A, n, batch, w, layout, fill, nthreads)


def potrs_il(L, B, n, nrhs, batch, w, layout: int = COL_MAJOR, fill: int = LOWER,
             nthreads: int = 1):
    return default().potrs_il(L, B, n, nrhs, batch, w, layout, fill, nthreads)


def getrf_getrs_il(A, B, n, nrhs, batch, w, layout: int = ROW_MAJOR, nthreads: int = 1,
                   tau: float = 1.0, ruda: int = 0, scale: int = 0):
    return default().getrf_getrs_il(A, B, n, nrhs, batch, w, layout, nthreads, tau, ruda,
                                    scale)


def potrf_potrs_il(A, B, n, nrhs, batch, w, layout: int = COL_MAJOR, fill: int = LOWER,
                   nthreads: int = 1, ruda: int = 0):
    return default().potrf_potrs_il(A, B, n, nrhs, batch, w, layout, fill, nthreads, ruda)


def _suffix(dtype) -> str:
    dt = np.dtype(dtype)
    if dt == np.float32:
        return "f32"
    if dt == np.float64:
        return "f64"
    raise TypeError(f"oracle supports float32/float64, not {dt}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)
