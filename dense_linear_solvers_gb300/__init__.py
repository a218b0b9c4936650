"""Batched small dense linear solvers for GB300 (sm_103a): Python binding.

This module only marshals arguments: it reads shapes, dtypes, device pointers and the
CUDA stream from torch tensors and calls the C ABI of ``libbsolve.so`` (declared in
``include/bsolve.h``) under the same names. Every step of every solve runs in the CUDA
kernels of that library; there is no CPU or PyTorch fallback. If the library has not
been built, importing works but every call raises.

Storage convention (raw storage tensors, as the C ABI sees memory):
  * A: (batch, n, n); row-major holds A itself, column-major holds A^T in memory;
  * B: (batch, n, nrhs) row-major, (batch, nrhs, n) column-major;
  * bdsv strips: (batch, nbr, bs, 3*bs), padded vector: (batch, (nbr + 2)*bs).
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libbsolve.so")

BS_OK, BS_ERR_INVALID_ARG, BS_ERR_UNSUPPORTED, BS_ERR_CUDA = 0, 1, 2, 3
BS_FP32, BS_FP64 = 0, 1
BS_ROW_MAJOR, BS_COL_MAJOR = 0, 1
BS_LOWER, BS_UPPER = 0, 1
BS_CONTRACT_DEFAULT, BS_CONTRACT_RUDA = 0, 1


class Options(ctypes.Structure):
    """bs_options: TDLS pivot threshold, the status contract and TDLS's row-major reading
    (see bsolve.h)."""
    _fields_ = [("pivot_threshold", ctypes.c_double), ("status_contract", ctypes.c_int),
                ("transposed_factor", ctypes.c_int), ("interleave", ctypes.c_int64),
                ("scaling", ctypes.c_int)]


ROW_MAJOR, COL_MAJOR = BS_ROW_MAJOR, BS_COL_MAJOR

EXPORTED = (
    "bs_getrf_getrs_batched", "bs_potrf_potrs_batched", "bs_bdsv_batched",
    "bs_getrf_batched", "bs_getrs_batched", "bs_potrf_batched", "bs_potrs_batched",
    "bs_bdsv_factor_batched", "bs_bdsv_solve_batched", "bs_bdmv_batched", "bs_bdmv2_batched",
    "bs_getrf_getrs_batched_ex", "bs_potrf_potrs_batched_ex",
    "bs_getrf_batched_ex", "bs_getrs_batched_ex", "bs_potrf_batched_ex", "bs_potrs_batched_ex",
    "bs_getrf_getrs_host_workspace", "bs_getrf_getrs_batched_host",
    "bs_potrf_potrs_host_workspace", "bs_potrf_potrs_batched_host",
    "bs_bdsv_host_workspace", "bs_bdsv_batched_host", "bs_getrf_getrs_batched_host_static",
    "bs_status_string", "bs_last_cuda_error", "bs_getrf_getrs_supported",
    "bs_potrf_potrs_supported", "bs_bdsv_supported", "bs_version",
)

_lock = threading.Lock()
_lib = None


class BsolveError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}"
                         + (f" (cuda error {lib().bs_last_cuda_error()})" if status == BS_ERR_CUDA
                            else ""))


def lib() -> ctypes.CDLL:
    """The loaded libbsolve.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "dense_linear_solvers_gb300._build.build() (or __graft_entry__.build()); "
                    "there is no fallback path")
            L = ctypes.CDLL(LIB_PATH)
            i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
            L.bs_getrf_getrs_batched.argtypes = [i32, i32, i32, i32, i64, vp, vp, vp, vp, vp]
            L.bs_getrf_getrs_batched.restype = i32
            L.bs_potrf_potrs_batched.argtypes = [i32, i32, i32, i32, i32, i64, vp, vp, vp, vp]
            L.bs_potrf_potrs_batched.restype = i32
            L.bs_bdsv_batched.argtypes = [i32, i32, i32, i64, vp, vp, vp, vp]
            L.bs_bdsv_batched.restype = i32
            L.bs_getrf_batched.argtypes = [i32, i32, i32, i64, vp, vp, vp, vp]
            L.bs_getrs_batched.argtypes = [i32, i32, i32, i32, i64, vp, vp, vp, vp]
            L.bs_potrf_batched.argtypes = [i32, i32, i32, i32, i64, vp, vp, vp]
            L.bs_potrs_batched.argtypes = [i32, i32, i32, i32, i32, i64, vp, vp, vp]
            L.bs_bdsv_factor_batched.argtypes = [i32, i32, i32, i64, vp, vp, vp]
            L.bs_bdsv_solve_batched.argtypes = [i32, i32, i32, i64, vp, vp, vp]
            L.bs_bdmv_batched.argtypes = [i32, i32, i32, i64, vp, vp, vp, vp]
            L.bs_bdmv2_batched.argtypes = [i32, i32, i32, i64, vp, vp, vp, vp, vp]
            L.bs_getrf_getrs_batched_ex.argtypes = [i32, i32, i32, i32, i64, vp, vp, vp, vp,
                                                    ctypes.POINTER(Options), vp]
            L.bs_potrf_potrs_batched_ex.argtypes = [i32, i32, i32, i32, i32, i64, vp, vp, vp,
                                                    ctypes.POINTER(Options), vp]
            L.bs_getrf_getrs_batched_ex.restype = i32
            L.bs_potrf_potrs_batched_ex.restype = i32
            opt = ctypes.POINTER(Options)
            L.bs_getrf_batched_ex.argtypes = [i32, i32, i32, i64, vp, vp, vp, opt, vp]
            L.bs_getrs_batched_ex.argtypes = [i32, i32, i32, i32, i64, vp, vp, vp, opt, vp]
            L.bs_potrf_batched_ex.argtypes = [i32, i32, i32, i32, i64, vp, vp, opt, vp]
            L.bs_potrs_batched_ex.argtypes = [i32, i32, i32, i32, i32, i64, vp, vp, opt, vp]
            for f in ("bs_getrf_batched_ex", "bs_getrs_batched_ex", "bs_potrf_batched_ex",
                      "bs_potrs_batched_ex"):
                getattr(L, f).restype = i32
            for name in ("bs_getrf_batched", "bs_getrs_batched", "bs_potrf_batched",
                         "bs_potrs_batched", "bs_bdsv_factor_batched", "bs_bdsv_solve_batched",
                         "bs_bdmv_batched", "bs_bdmv2_batched"):
                getattr(L, name).restype = i32
            sz = ctypes.c_size_t
            L.bs_getrf_getrs_host_workspace.argtypes = [i32, i32, i32, i64]
            L.bs_potrf_potrs_host_workspace.argtypes = [i32, i32, i32, i64]
            L.bs_bdsv_host_workspace.argtypes = [i32, i32, i32, i64]
            for name in ("bs_getrf_getrs_host_workspace", "bs_potrf_potrs_host_workspace",
                         "bs_bdsv_host_workspace"):
                getattr(L, name).restype = sz
            L.bs_getrf_getrs_batched_host.argtypes = [i32, i32, i32, i32, i64, vp, vp, vp, vp,
                                                      vp, sz, i64, vp, vp]
            L.bs_potrf_potrs_batched_host.argtypes = [i32, i32, i32, i32, i32, i64, vp, vp, vp,
                                                      vp, sz, i64, vp, vp]
            L.bs_bdsv_batched_host.argtypes = [i32, i32, i32, i64, vp, vp, vp, vp, sz, i64, vp,
                                               vp]
            L.bs_getrf_getrs_batched_host_static.argtypes = [i32, i32, i32, i32, i64, vp, vp,
                                                             vp, vp, i64, vp, vp]
            for name in ("bs_getrf_getrs_batched_host", "bs_potrf_potrs_batched_host",
                         "bs_bdsv_batched_host", "bs_getrf_getrs_batched_host_static"):
                getattr(L, name).restype = i32
            L.bs_status_string.argtypes = [i32]
            L.bs_status_string.restype = ctypes.c_char_p
            L.bs_last_cuda_error.argtypes = []
            L.bs_last_cuda_error.restype = i32
            L.bs_getrf_getrs_supported.argtypes = [i32, i32, i32, i32]
            L.bs_getrf_getrs_supported.restype = i32
            L.bs_potrf_potrs_supported.argtypes = [i32, i32, i32, i32, i32]
            L.bs_potrf_potrs_supported.restype = i32
            L.bs_bdsv_supported.argtypes = [i32, i32, i32]
            L.bs_bdsv_supported.restype = i32
            L.bs_version.argtypes = []
            L.bs_version.restype = i32
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().bs_status_string(int(status)).decode()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return BS_FP32
    if t.dtype == torch.float64:
        return BS_FP64
    raise TypeError(f"unsupported dtype {t.dtype}: float32 or float64")


def _ptr(t) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError("bsolve operands are device tensors (torch CUDA tensors)")
    if not t.is_contiguous():
        raise ValueError("bsolve operands must be contiguous")
    return t.data_ptr()


def _expect(t, name: str, dtype, numel: int) -> None:
    """An operand's element type and element count, checked before its pointer is taken:
    the library sees only pointers and sizes, so a tensor of another type or size would be
    read as if it were the expected one. None passes (the library reports the null)."""
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if t.numel() != numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")


def _dense(A, B, layout: int):
    """(batch, n, nrhs) of a dense call, B checked against A: A is (batch, n, n); B is
    (batch, n, nrhs) in row-major storage, (batch, nrhs, n) in column-major, of A's dtype.
    B None: a factor call (nrhs 0)."""
    if A.dim() != 3 or A.shape[1] != A.shape[2]:
        raise ValueError(f"A: shape {tuple(A.shape)}, expected (batch, n, n)")
    batch, n = A.shape[0], A.shape[1]
    if B is None:
        return batch, n, 0
    if B.dim() != 3 or B.shape[0] != batch or B.shape[1 if layout == ROW_MAJOR else 2] != n:
        want = "(batch, n, nrhs)" if layout == ROW_MAJOR else "(batch, nrhs, n)"
        raise ValueError(f"B: shape {tuple(B.shape)}, expected {want} with batch {batch}, n {n}")
    if B.dtype != A.dtype:
        raise TypeError(f"B: dtype {B.dtype}, expected A's {A.dtype}")
    return batch, n, (B.shape[2] if layout == ROW_MAJOR else B.shape[1])


def _pivots(ipiv, info, batch: int, n: int, held: int | None = None) -> None:
    # ipiv: n int32 per system (held systems of an interleaved batch); info: one per system
    import torch
    _expect(ipiv, "ipiv", torch.int32, (batch if held is None else held) * n)
    _expect(info, "info", torch.int32, batch)


def _strips(strips, vectors, info):
    """(batch, nbr, bs) of a block-tridiagonal call: strips (batch, nbr, bs, 3*bs); each
    padded vector (nbr + 2) * bs per system, of the strips' dtype; info one int32 each."""
    import torch
    if strips.dim() != 4 or strips.shape[3] != 3 * strips.shape[2]:
        raise ValueError(f"strips: shape {tuple(strips.shape)}, expected (batch, nbr, bs, 3*bs)")
    batch, nbr, bsz = strips.shape[0], strips.shape[1], strips.shape[2]
    for name, v in vectors:
        _expect(v, name, strips.dtype, batch * (nbr + 2) * bsz)
    if info is not None:
        _expect(info, "info", torch.int32, batch)
    return batch, nbr, bsz


def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, what: str) -> None:
    if status != BS_OK:
        raise BsolveError(status, what)


def bs_getrf_getrs_batched(A, B, ipiv, info, layout: int = ROW_MAJOR, stream=None) -> None:
    """LU with partial pivoting + solve of A[s] X = B[s], in place (see bsolve.h)."""
    batch, n, nrhs = _dense(A, B, layout)
    _pivots(ipiv, info, batch, n)
    st = lib().bs_getrf_getrs_batched(_dtype_code(A), layout, n, nrhs, batch, _ptr(A), _ptr(B),
                                      _ptr(ipiv), _ptr(info), _stream(stream))
    _check(st, "bs_getrf_getrs_batched")


def bs_potrf_potrs_batched(A, B, info, layout: int = COL_MAJOR, fill: int = BS_LOWER,
                           stream=None) -> None:
    """Cholesky + solve of SPD systems, in place (see bsolve.h)."""
    batch, n, nrhs = _dense(A, B, layout)
    _pivots(None, info, batch, n)
    st = lib().bs_potrf_potrs_batched(_dtype_code(A), layout, fill, n, nrhs, batch, _ptr(A),
                                      _ptr(B), _ptr(info), _stream(stream))
    _check(st, "bs_potrf_potrs_batched")


def bs_bdsv_batched(strips, x_padded, info, stream=None) -> None:
    """Block-tridiagonal block-Cholesky solve, in place (see bsolve.h)."""
    batch, nbr, bs = _strips(strips, [("x_padded", x_padded)], info)
    st = lib().bs_bdsv_batched(_dtype_code(strips), nbr, bs, batch, _ptr(strips), _ptr(x_padded),
                               _ptr(info), _stream(stream))
    _check(st, "bs_bdsv_batched")


# --------------------------------------------- factor once, solve per right-hand side
def bs_getrf_batched(A, ipiv, info, layout: int = ROW_MAJOR, stream=None) -> None:
    """LU with partial pivoting alone, in place: A <- L\\U, ipiv, info (see bsolve.h)."""
    batch, n, _ = _dense(A, None, layout)
    _pivots(ipiv, info, batch, n)
    st = lib().bs_getrf_batched(_dtype_code(A), layout, n, batch, _ptr(A), _ptr(ipiv), _ptr(info),
                                _stream(stream))
    _check(st, "bs_getrf_batched")


def bs_getrs_batched(LU, ipiv, B, layout: int = ROW_MAJOR, stream=None) -> None:
    """Solve with a getrf factor: B <- X (see bsolve.h)."""
    batch, n, nrhs = _dense(LU, B, layout)
    _pivots(ipiv, None, batch, n)
    st = lib().bs_getrs_batched(_dtype_code(LU), layout, n, nrhs, batch, _ptr(LU), _ptr(ipiv),
                                _ptr(B), _stream(stream))
    _check(st, "bs_getrs_batched")


def bs_potrf_batched(A, info, layout: int = COL_MAJOR, fill: int = BS_LOWER, stream=None) -> None:
    """Cholesky alone, in place: the lower triangle of A <- L, info (see bsolve.h)."""
    batch, n, _ = _dense(A, None, layout)
    _pivots(None, info, batch, n)
    st = lib().bs_potrf_batched(_dtype_code(A), layout, fill, n, batch, _ptr(A), _ptr(info),
                                _stream(stream))
    _check(st, "bs_potrf_batched")


def bs_potrs_batched(L, B, layout: int = COL_MAJOR, fill: int = BS_LOWER, stream=None) -> None:
    """Solve with a potrf factor: B <- X (see bsolve.h)."""
    batch, n, nrhs = _dense(L, B, layout)
    st = lib().bs_potrs_batched(_dtype_code(L), layout, fill, n, nrhs, batch, _ptr(L), _ptr(B),
                                _stream(stream))
    _check(st, "bs_potrs_batched")


def bs_bdsv_factor_batched(strips, info, stream=None) -> None:
    """Block-Cholesky factor sweep alone, in place on the strips (see bsolve.h)."""
    batch, nbr, bs = _strips(strips, [], info)
    st = lib().bs_bdsv_factor_batched(_dtype_code(strips), nbr, bs, batch, _ptr(strips),
                                      _ptr(info), _stream(stream))
    _check(st, "bs_bdsv_factor_batched")


def bs_bdsv_solve_batched(strips, x_padded, stream=None) -> None:
    """Forward/backward block substitution with factored strips, in place on x (see
    bsolve.h)."""
    batch, nbr, bs = _strips(strips, [("x_padded", x_padded)], None)
    st = lib().bs_bdsv_solve_batched(_dtype_code(strips), nbr, bs, batch, _ptr(strips),
                                     _ptr(x_padded), _stream(stream))
    _check(st, "bs_bdsv_solve_batched")


def bs_bdmv_batched(strips, x_padded, y_padded, stream=None) -> None:
    """Block-tridiagonal matvec: the interior of y_padded <- A x (see bsolve.h)."""
    batch, nbr, bs = _strips(strips, [("x_padded", x_padded), ("y_padded", y_padded)], None)
    st = lib().bs_bdmv_batched(_dtype_code(strips), nbr, bs, batch, _ptr(strips), _ptr(x_padded),
                               _ptr(y_padded), _stream(stream))
    _check(st, "bs_bdmv_batched")


def bs_bdmv2_batched(strips, x_padded, y_padded, y2_padded, stream=None) -> None:
    """The matvec stored into two padded outputs in one pass (see bsolve.h)."""
    batch, nbr, bs = _strips(strips, [("x_padded", x_padded), ("y_padded", y_padded),
                                      ("y2_padded", y2_padded)], None)
    st = lib().bs_bdmv2_batched(_dtype_code(strips), nbr, bs, batch, _ptr(strips),
                                _ptr(x_padded), _ptr(y_padded), _ptr(y2_padded),
                                _stream(stream))
    _check(st, "bs_bdmv2_batched")


# --------------------------------------------------------------- contract variants
def _il_shape(A, B, ipiv, info, layout, interleave, shape):
    """(batch, n, nrhs) of a contract-variant call, the operands checked. The plain batched
    layout: from the tensors' shapes, as the plain calls. Interleaved (interleave = W > 1):
    given as shape; A, B and ipiv are flat and hold whole blocks, ceil(batch / W) * W
    systems each; info one entry per system."""
    if interleave > 1:
        if shape is None:
            raise ValueError("an interleaved batch needs shape=(batch, n, nrhs)")
        batch, n, nrhs = (int(v) for v in shape)
        held = -(-batch // interleave) * interleave
        _dtype_code(A)
        _expect(A, "A", A.dtype, held * n * n)
        _expect(B, "B", A.dtype, held * n * nrhs)
        _pivots(ipiv, info, batch, n, held)
        return batch, n, nrhs
    batch, n, nrhs = _dense(A, B, layout)
    _pivots(ipiv, info, batch, n)
    return batch, n, nrhs


def bs_getrf_getrs_batched_ex(A, B, ipiv, info, layout: int = ROW_MAJOR,
                              pivot_threshold: float = 1.0,
                              status_contract: int = BS_CONTRACT_DEFAULT,
                              transposed_factor: int = 0, interleave: int = 0, shape=None,
                              scaling: int = 0, stream=None) -> None:
    """LU + solve with TDLS threshold pivoting, the RUDA status contract, TDLS's
    row-major reading (factor of A^T and the mirror solve), or an interleaved batched
    layout (A, B, ipiv flat; shape=(batch, n, nrhs)), or RUDA's max-abs scaling."""
    batch, n, nrhs = _il_shape(A, B, ipiv, info, layout, interleave, shape)
    opts = Options(float(pivot_threshold), int(status_contract), int(transposed_factor),
                   int(interleave), int(scaling))
    st = lib().bs_getrf_getrs_batched_ex(_dtype_code(A), layout, n, nrhs, batch, _ptr(A), _ptr(B),
                                         _ptr(ipiv), _ptr(info), ctypes.byref(opts),
                                         _stream(stream))
    _check(st, "bs_getrf_getrs_batched_ex")


def bs_potrf_potrs_batched_ex(A, B, info, layout: int = COL_MAJOR, fill: int = BS_LOWER,
                              status_contract: int = BS_CONTRACT_DEFAULT, interleave: int = 0,
                              shape=None, stream=None) -> None:
    """Cholesky + solve under the RUDA status contract, or on an interleaved batched
    layout (A, B flat; shape=(batch, n, nrhs))."""
    batch, n, nrhs = _il_shape(A, B, None, info, layout, interleave, shape)
    opts = Options(1.0, int(status_contract), 0, int(interleave), 0)
    st = lib().bs_potrf_potrs_batched_ex(_dtype_code(A), layout, fill, n, nrhs, batch, _ptr(A),
                                         _ptr(B), _ptr(info), ctypes.byref(opts), _stream(stream))
    _check(st, "bs_potrf_potrs_batched_ex")


def _factor_shape(shape):
    # a factor call's interleaved shape: (batch, n) or (batch, n, anything)
    return None if shape is None else (shape[0], shape[1], 0)


def bs_getrf_batched_ex(A, ipiv, info, layout: int = ROW_MAJOR, pivot_threshold: float = 1.0,
                        transposed_factor: int = 0, interleave: int = 0, shape=None,
                        status_contract: int = BS_CONTRACT_DEFAULT, scaling: int = 0,
                        stream=None) -> None:
    """getrf alone with the threshold, the row-major reading or an interleaved layout (A,
    ipiv flat; shape=(batch, n)): the fused _ex call's factor (see bsolve.h)."""
    batch, n, _ = _il_shape(A, None, ipiv, info, layout, interleave, _factor_shape(shape))
    opts = Options(float(pivot_threshold), int(status_contract), int(transposed_factor),
                   int(interleave), int(scaling))
    st = lib().bs_getrf_batched_ex(_dtype_code(A), layout, n, batch, _ptr(A), _ptr(ipiv),
                                   _ptr(info), ctypes.byref(opts), _stream(stream))
    _check(st, "bs_getrf_batched_ex")


def bs_getrs_batched_ex(LU, ipiv, B, layout: int = ROW_MAJOR, transposed_factor: int = 0,
                        interleave: int = 0, shape=None, pivot_threshold: float = 1.0,
                        status_contract: int = BS_CONTRACT_DEFAULT, scaling: int = 0,
                        stream=None) -> None:
    """getrs with a bs_getrf_batched_ex factor: the mirror solve of the row-major reading,
    or an interleaved layout (LU, ipiv, B flat; shape=(batch, n, nrhs)) (see bsolve.h)."""
    batch, n, nrhs = _il_shape(LU, B, ipiv, None, layout, interleave, shape)
    opts = Options(float(pivot_threshold), int(status_contract), int(transposed_factor),
                   int(interleave), int(scaling))
    st = lib().bs_getrs_batched_ex(_dtype_code(LU), layout, n, nrhs, batch, _ptr(LU), _ptr(ipiv),
                                   _ptr(B), ctypes.byref(opts), _stream(stream))
    _check(st, "bs_getrs_batched_ex")


def bs_potrf_batched_ex(A, info, layout: int = COL_MAJOR, fill: int = BS_LOWER,
                        interleave: int = 0, shape=None,
                        status_contract: int = BS_CONTRACT_DEFAULT, transposed_factor: int = 0,
                        stream=None) -> None:
    """potrf alone on an interleaved layout (A flat; shape=(batch, n)) (see bsolve.h)."""
    batch, n, _ = _il_shape(A, None, None, info, layout, interleave, _factor_shape(shape))
    opts = Options(1.0, int(status_contract), int(transposed_factor), int(interleave), 0)
    st = lib().bs_potrf_batched_ex(_dtype_code(A), layout, fill, n, batch, _ptr(A), _ptr(info),
                                   ctypes.byref(opts), _stream(stream))
    _check(st, "bs_potrf_batched_ex")


def bs_potrs_batched_ex(L, B, layout: int = COL_MAJOR, fill: int = BS_LOWER,
                        interleave: int = 0, shape=None,
                        status_contract: int = BS_CONTRACT_DEFAULT, stream=None) -> None:
    """potrs with a bs_potrf_batched_ex factor on an interleaved layout (L, B flat;
    shape=(batch, n, nrhs)) (see bsolve.h)."""
    batch, n, nrhs = _il_shape(L, B, None, None, layout, interleave, shape)
    opts = Options(1.0, int(status_contract), 0, int(interleave), 0)
    st = lib().bs_potrs_batched_ex(_dtype_code(L), layout, fill, n, nrhs, batch, _ptr(L), _ptr(B),
                                   ctypes.byref(opts), _stream(stream))
    _check(st, "bs_potrs_batched_ex")


# ------------------------------------------------------------ host-resident batches
def _host_ptr(t) -> int:
    if t.is_cuda:
        raise ValueError("the *_host calls take host (CPU) tensors; pinned memory overlaps")
    if not t.is_contiguous():
        raise ValueError("bsolve operands must be contiguous")
    return t.data_ptr()


class HostPlan:
    """Device workspace and the two streams of the *_host calls (plumbing: the workspace
    is a torch CUDA tensor sized by the library's query; the library allocates nothing)."""

    def __init__(self, work_bytes: int, streams=None):
        import torch
        self.work = torch.empty(max(int(work_bytes), 1), dtype=torch.uint8, device="cuda")
        self.streams = tuple(streams) if streams else (torch.cuda.Stream(), torch.cuda.Stream())

    def synchronize(self):
        for st in self.streams:
            st.synchronize()


def getrf_getrs_host_plan(dtype_code: int, n: int, nrhs: int, chunk: int, streams=None):
    return HostPlan(lib().bs_getrf_getrs_host_workspace(dtype_code, n, nrhs, chunk), streams)


def potrf_potrs_host_plan(dtype_code: int, n: int, nrhs: int, chunk: int, streams=None):
    return HostPlan(lib().bs_potrf_potrs_host_workspace(dtype_code, n, nrhs, chunk), streams)


def bdsv_host_plan(dtype_code: int, nbr: int, bsz: int, chunk: int, streams=None):
    return HostPlan(lib().bs_bdsv_host_workspace(dtype_code, nbr, bsz, chunk), streams)


def bs_getrf_getrs_batched_host(A, B, ipiv, info, layout: int = ROW_MAJOR, chunk: int = 8192,
                                plan: HostPlan | None = None, sync: bool = True) -> HostPlan:
    """LU + solve on host tensors, in place, copied in and out by chunks on two streams."""
    batch, n, nrhs = _dense(A, B, layout)
    _pivots(ipiv, info, batch, n)
    plan = plan or getrf_getrs_host_plan(_dtype_code(A), n, nrhs, chunk)
    st = lib().bs_getrf_getrs_batched_host(
        _dtype_code(A), layout, n, nrhs, batch, _host_ptr(A), _host_ptr(B), _host_ptr(ipiv),
        _host_ptr(info), plan.work.data_ptr(), plan.work.numel(), chunk,
        _stream(plan.streams[0]), _stream(plan.streams[1]))
    _check(st, "bs_getrf_getrs_batched_host")
    if sync:
        plan.synchronize()
    return plan


def bs_potrf_potrs_batched_host(A, B, info, layout: int = COL_MAJOR, fill: int = BS_LOWER,
                                chunk: int = 8192, plan: HostPlan | None = None,
                                sync: bool = True) -> HostPlan:
    """Cholesky + solve on host tensors, in place, by chunks on two streams."""
    batch, n, nrhs = _dense(A, B, layout)
    _pivots(None, info, batch, n)
    plan = plan or potrf_potrs_host_plan(_dtype_code(A), n, nrhs, chunk)
    st = lib().bs_potrf_potrs_batched_host(
        _dtype_code(A), layout, fill, n, nrhs, batch, _host_ptr(A), _host_ptr(B),
        _host_ptr(info), plan.work.data_ptr(), plan.work.numel(), chunk,
        _stream(plan.streams[0]), _stream(plan.streams[1]))
    _check(st, "bs_potrf_potrs_batched_host")
    if sync:
        plan.synchronize()
    return plan


def bs_bdsv_batched_host(strips, x_padded, info, chunk: int = 2048,
                         plan: HostPlan | None = None, sync: bool = True) -> HostPlan:
    """Block-tridiagonal solve on host tensors, in place, by chunks on two streams."""
    batch, nbr, bsz = _strips(strips, [("x_padded", x_padded)], info)
    plan = plan or bdsv_host_plan(_dtype_code(strips), nbr, bsz, chunk)
    st = lib().bs_bdsv_batched_host(
        _dtype_code(strips), nbr, bsz, batch, _host_ptr(strips), _host_ptr(x_padded),
        _host_ptr(info), plan.work.data_ptr(), plan.work.numel(), chunk,
        _stream(plan.streams[0]), _stream(plan.streams[1]))
    _check(st, "bs_bdsv_batched_host")
    if sync:
        plan.synchronize()
    return plan


def bs_getrf_getrs_batched_host_static(A, B, ipiv, info, layout: int = ROW_MAJOR,
                                       chunk: int = 16384, streams=None,
                                       sync: bool = True):
    """bs_getrf_getrs_batched_host on the library's static device scratch (no workspace
    argument; see bsolve.h for the one-call-at-a-time rule). Returns the two streams."""
    import torch
    batch, n, nrhs = _dense(A, B, layout)
    _pivots(ipiv, info, batch, n)
    streams = tuple(streams) if streams else (torch.cuda.Stream(), torch.cuda.Stream())
    st = lib().bs_getrf_getrs_batched_host_static(
        _dtype_code(A), layout, n, nrhs, batch, _host_ptr(A), _host_ptr(B), _host_ptr(ipiv),
        _host_ptr(info), chunk, _stream(streams[0]), _stream(streams[1]))
    _check(st, "bs_getrf_getrs_batched_host_static")
    if sync:
        for s_ in streams:
            s_.synchronize()
    return streams
