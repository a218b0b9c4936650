"""The C ABI on the host: the library loads, exports every symbol bsolve.h declares,
and rejects bad arguments before launching anything (no GPU needed: none of these calls
reaches the CUDA runtime)."""
import ctypes
import os
import re

import numpy as np
import pytest

import dense_linear_solvers_gb300 as bs
from dense_linear_solvers_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "bsolve.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return bs.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"BS_API\s+[\w\s\*]+?\b(bs_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for must in ("bs_getrf_getrs_batched", "bs_potrf_potrs_batched", "bs_bdsv_batched",
                 "bs_status_string"):
        assert must in names
    assert set(names) == set(bs.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        ctypes.cast(getattr(lib, name), ctypes.c_void_p)


def test_status_strings(lib):
    assert bs.status_string(bs.BS_OK) == "BS_OK"
    assert bs.status_string(bs.BS_ERR_UNSUPPORTED) == "BS_ERR_UNSUPPORTED"
    assert bs.status_string(99) == "BS_UNKNOWN_STATUS"
    assert lib.bs_version() >= 100
    assert lib.bs_last_cuda_error() == 0


def test_supported_queries(lib):
    assert lib.bs_getrf_getrs_supported(bs.BS_FP32, bs.BS_ROW_MAJOR, 16, 4) == 1
    assert lib.bs_getrf_getrs_supported(bs.BS_FP64, bs.BS_COL_MAJOR, 64, 8) == 1
    assert lib.bs_getrf_getrs_supported(bs.BS_FP64, bs.BS_ROW_MAJOR, 129, 1) == 0
    assert lib.bs_getrf_getrs_supported(bs.BS_FP64, bs.BS_ROW_MAJOR, 8, 9) == 1
    assert lib.bs_getrf_getrs_supported(bs.BS_FP64, bs.BS_ROW_MAJOR, 8, 65537) == 0
    assert lib.bs_getrf_getrs_supported(2, bs.BS_ROW_MAJOR, 8, 1) == 0
    assert lib.bs_potrf_potrs_supported(bs.BS_FP64, bs.BS_COL_MAJOR, bs.BS_LOWER, 32, 1) == 1
    assert lib.bs_potrf_potrs_supported(bs.BS_FP64, bs.BS_COL_MAJOR, bs.BS_UPPER, 32, 1) == 1
    assert lib.bs_potrf_potrs_supported(bs.BS_FP64, bs.BS_COL_MAJOR, 2, 32, 1) == 0
    assert lib.bs_bdsv_supported(bs.BS_FP64, 32, 8) == 1
    assert lib.bs_bdsv_supported(bs.BS_FP64, 32, 9) == 0


COL = bs.BS_COL_MAJOR
FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below returns early


def test_lu_argument_errors(lib):
    f = lib.bs_getrf_getrs_batched
    assert f(bs.BS_FP32, 0, 16, 4, 0, None, None, None, None, None) == bs.BS_OK  # empty batch
    assert f(bs.BS_FP32, 0, 16, 4, -1, FAKE, FAKE, FAKE, FAKE, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, -3, 4, 5, FAKE, FAKE, FAKE, FAKE, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 129, 4, 5, FAKE, FAKE, FAKE, FAKE, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 0, 4, 5, FAKE, FAKE, FAKE, FAKE, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 65537, 5, FAKE, FAKE, FAKE, FAKE, None) == bs.BS_ERR_UNSUPPORTED
    assert f(7, 0, 16, 4, 5, FAKE, FAKE, FAKE, FAKE, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 5, 16, 4, 5, FAKE, FAKE, FAKE, FAKE, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 4, 5, None, FAKE, FAKE, FAKE, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, FAKE, FAKE, None, FAKE, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, FAKE + 4, FAKE, FAKE, FAKE, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP64, 1, 16, 4, 5, FAKE, FAKE + 8, FAKE, FAKE, None) == bs.BS_ERR_INVALID_ARG


def test_chol_argument_errors(lib):
    f = lib.bs_potrf_potrs_batched
    assert f(bs.BS_FP64, 1, 0, 32, 1, 0, None, None, None, None) == bs.BS_OK
    assert f(bs.BS_FP64, 1, 2, 32, 1, 5, FAKE, FAKE, FAKE, None) == bs.BS_ERR_UNSUPPORTED  # bad fill
    assert f(bs.BS_FP64, 1, 0, 32, 1, 5, FAKE, None, FAKE, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP64, 1, 0, 32, 1, 5, FAKE, FAKE, FAKE + 2, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP64, 1, 0, 32, -1, 5, FAKE, FAKE, FAKE, None) == bs.BS_ERR_INVALID_ARG


def test_bdsv_argument_errors(lib):
    f = lib.bs_bdsv_batched
    assert f(bs.BS_FP64, 32, 8, 0, None, None, None, None) == bs.BS_OK
    assert f(bs.BS_FP64, 32, 9, 4, FAKE, FAKE, FAKE, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP64, 0, 8, 4, FAKE, FAKE, FAKE, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP64, -1, 8, 4, FAKE, FAKE, FAKE, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP64, 32, 8, 4, FAKE, None, FAKE, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP64, 32, 8, 4, FAKE, FAKE + 8, FAKE, None) == bs.BS_ERR_INVALID_ARG


def test_split_argument_errors(lib):
    """The factor and solve halves check their arguments like the fused calls, and the
    solve calls refuse an output that overlaps a read-only input."""
    A, B, P, I = FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000
    f = lib.bs_getrf_batched
    assert f(bs.BS_FP32, 0, 16, 0, None, None, None, None) == bs.BS_OK
    assert f(bs.BS_FP32, 0, 129, 5, A, P, I, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, -1, 5, A, P, I, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 5, A, None, I, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 5, A + 4, P, I, None) == bs.BS_ERR_INVALID_ARG
    f = lib.bs_getrs_batched
    assert f(bs.BS_FP32, 0, 16, 4, 0, None, None, None, None) == bs.BS_OK
    assert f(bs.BS_FP32, 0, 16, 65537, 5, A, P, B, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, P, None, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, P, A + 16, None) == bs.BS_ERR_INVALID_ARG  # B over LU
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, P, P, None) == bs.BS_ERR_INVALID_ARG       # B over ipiv
    f = lib.bs_potrf_batched
    assert f(bs.BS_FP64, 1, 0, 32, 0, None, None, None) == bs.BS_OK
    assert f(bs.BS_FP64, 1, 3, 32, 5, A, I, None) == bs.BS_ERR_UNSUPPORTED  # bad fill
    assert f(bs.BS_FP64, 1, 0, 32, 5, A, None, None) == bs.BS_ERR_INVALID_ARG
    f = lib.bs_potrs_batched
    assert f(bs.BS_FP64, 1, 0, 32, 1, 0, None, None, None) == bs.BS_OK
    assert f(bs.BS_FP64, 1, 0, 32, 1, 5, A, A, None) == bs.BS_ERR_INVALID_ARG       # B over L
    assert f(bs.BS_FP64, 1, 0, 32, 0, 5, A, B, None) == bs.BS_ERR_UNSUPPORTED
    f = lib.bs_bdsv_factor_batched
    assert f(bs.BS_FP64, 32, 8, 0, None, None, None) == bs.BS_OK
    assert f(bs.BS_FP64, 32, 9, 4, A, I, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP64, 32, 8, 4, A, None, None) == bs.BS_ERR_INVALID_ARG
    f = lib.bs_bdsv_solve_batched
    assert f(bs.BS_FP64, 32, 8, 0, None, None, None) == bs.BS_OK
    assert f(bs.BS_FP64, 32, 8, 4, A, A + 64, None) == bs.BS_ERR_INVALID_ARG        # x over strips
    assert f(bs.BS_FP64, 32, 8, 4, A, B + 8, None) == bs.BS_ERR_INVALID_ARG         # misaligned
    f = lib.bs_bdmv_batched
    assert f(bs.BS_FP64, 32, 8, 0, None, None, None, None) == bs.BS_OK
    assert f(bs.BS_FP64, 32, 0, 4, A, B, P, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP64, 32, 8, 4, A, B, None, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP64, 32, 8, 4, A, B, B + 16, None) == bs.BS_ERR_INVALID_ARG     # y over x
    assert f(bs.BS_FP64, 32, 8, 4, A, B, A, None) == bs.BS_ERR_INVALID_ARG          # y over strips
    f = lib.bs_bdmv2_batched
    assert f(bs.BS_FP64, 32, 8, 0, None, None, None, None, None) == bs.BS_OK
    assert f(bs.BS_FP64, 32, 0, 4, A, B, P, I, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP64, 32, 8, 4, A, B, P, None, None) == bs.BS_ERR_INVALID_ARG    # no y2
    assert f(bs.BS_FP64, 32, 8, 4, A, B, P, I + 8, None) == bs.BS_ERR_INVALID_ARG   # misaligned
    assert f(bs.BS_FP64, 32, 8, 4, A, B, P, P + 16, None) == bs.BS_ERR_INVALID_ARG  # y2 over y
    assert f(bs.BS_FP64, 32, 8, 4, A, B, P, A, None) == bs.BS_ERR_INVALID_ARG       # y2 over strips
    assert f(bs.BS_FP64, 32, 8, 4, A, B, P, B, None) == bs.BS_ERR_INVALID_ARG       # y2 over x


def test_contract_variant_argument_errors(lib):
    """Options are checked before anything else: a threshold outside (0, 1] or an unknown
    contract is an argument error; options other than the defaults hold 8 right-hand
    sides at most."""
    import ctypes
    A, B, P, I = FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000
    f = lib.bs_getrf_getrs_batched_ex
    o = lambda tau, c: ctypes.byref(bs.Options(tau, c))  # noqa: E731
    assert f(bs.BS_FP32, 0, 16, 4, 0, None, None, None, None, o(0.5, 0), None) == bs.BS_OK
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, o(0.0, 0), None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, o(1.5, 0), None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, o(float("nan"), 0), None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, o(1.0, 7), None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 9, 5, A, B, P, I, o(0.5, 0), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 129, 4, 5, A, B, P, I, o(0.5, 1), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 4, 5, None, B, P, I, o(0.5, 1), None) == bs.BS_ERR_INVALID_ARG
    g = lib.bs_potrf_potrs_batched_ex
    assert g(bs.BS_FP64, 1, 0, 32, 1, 0, None, None, None, o(1.0, 1), None) == bs.BS_OK
    assert g(bs.BS_FP64, 1, 0, 32, 1, 5, A, B, I, o(1.0, 2), None) == bs.BS_ERR_INVALID_ARG
    assert g(bs.BS_FP64, 1, 0, 32, 9, 5, A, B, I, o(1.0, 1), None) == bs.BS_ERR_UNSUPPORTED
    assert g(bs.BS_FP64, 1, 0, 32, 1, 5, A, None, I, o(1.0, 1), None) == bs.BS_ERR_INVALID_ARG
    # TDLS's row-major reading: 0 or 1, not with the RUDA contract, up to 65536
    # right-hand sides (a factor launch and a solve launch); the size of bs_options is
    # a double and two ints
    assert ctypes.sizeof(bs.Options) == 32
    m = lambda tau, c, t: ctypes.byref(bs.Options(tau, c, t))  # noqa: E731
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, m(1.0, 0, 2), None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, m(1.0, 1, 1), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 129, 4, 5, A, B, P, I, m(1.0, 0, 1), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 65537, 5, A, B, P, I, m(0.5, 0, 1), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 9, 0, None, None, None, None, m(0.5, 0, 1), None) == bs.BS_OK
    assert f(bs.BS_FP32, 0, 16, 9, 5, A, B, None, I, m(0.5, 0, 1), None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 9, 5, A + 4, B, P, I, m(1.0, 0, 1), None) == bs.BS_ERR_INVALID_ARG
    # the interleaved batched layout: W >= 0; with W > 1 at most 8 right-hand sides, except
    # under the row-major reading (a solve launch of its own)
    w = lambda tau, c, t, il: ctypes.byref(bs.Options(tau, c, t, il))  # noqa: E731
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, w(1.0, 0, 0, -1), None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 9, 5, A, B, P, I, w(0.5, 0, 0, 32), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 9, 5, A, B, P, I, w(1.0, 1, 0, 32), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 9, 5, A, B, P, I + 4, w(1.0, 0, 1, 32), None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 65537, 5, A, B, P, I, w(1.0, 0, 1, 32), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, w(1.0, 1, 1, 32), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 9, 5, A, B, P, I, w(1.0, 0, 0, 32), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 129, 4, 5, A, B, P, I, w(1.0, 0, 0, 32), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 4, 0, None, None, None, None, w(1.0, 0, 0, 32), None) == bs.BS_OK
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P + 8, I, w(1.0, 0, 0, 32), None) == bs.BS_ERR_INVALID_ARG
    assert g(bs.BS_FP64, 1, 0, 32, 1, 5, A, B, I, w(1.0, 0, 0, -3), None) == bs.BS_ERR_INVALID_ARG
    assert g(bs.BS_FP64, 1, 0, 32, 9, 5, A, B, I, w(1.0, 1, 0, 64), None) == bs.BS_ERR_UNSUPPORTED
    assert g(bs.BS_FP64, 1, 0, 32, 1, 5, A, B, I, w(1.0, 0, 1, 0), None) == bs.BS_ERR_UNSUPPORTED
    assert g(bs.BS_FP64, 1, 0, 32, 9, 5, A, B, I, w(1.0, 0, 0, 64), None) == bs.BS_ERR_UNSUPPORTED
    assert g(bs.BS_FP64, 1, 0, 32, 1, 0, None, None, None, w(1.0, 0, 0, 64), None) == bs.BS_OK
    # RUDA's max-abs scaling: 0 or 1, LU only (the row-major reading included)
    sc = lambda tau, c, t, il, k: ctypes.byref(bs.Options(tau, c, t, il, k))  # noqa: E731
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, sc(1.0, 0, 0, 0, 2), None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, A + 4, B, P, I, sc(1.0, 0, 1, 0, 1), None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 129, 4, 5, A, B, P, I, sc(1.0, 0, 1, 8, 1), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 9, 5, A, B, P, I, sc(1.0, 0, 0, 0, 1), None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, 4, 0, None, None, None, None, sc(1.0, 0, 0, 0, 1), None) == bs.BS_OK
    assert g(bs.BS_FP64, 1, 0, 32, 1, 5, A, B, I, sc(1.0, 0, 0, 0, 1), None) == bs.BS_ERR_UNSUPPORTED
    assert g(bs.BS_FP64, 1, 0, 32, 1, 5, A, B, I, sc(1.0, 0, 0, 0, 3), None) == bs.BS_ERR_INVALID_ARG


def test_split_calls_with_options_argument_errors(lib):
    """The split _ex calls check their options as the fused _ex calls do; the RUDA
    contract and the scaling stay with the fused calls, Cholesky takes no LU option;
    interleaved operands hold whole blocks (5 systems in blocks of 4: room for 8)."""
    import ctypes
    A, B, P, I = FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000
    o = lambda tau=1.0, c=0, t=0, il=0, k=0: ctypes.byref(bs.Options(tau, c, t, il, k))  # noqa: E731
    gf, gs = lib.bs_getrf_batched_ex, lib.bs_getrs_batched_ex
    pf, ps = lib.bs_potrf_batched_ex, lib.bs_potrs_batched_ex
    assert gf(bs.BS_FP64, 0, 8, 5, A, P, I, o(tau=0.0), None) == bs.BS_ERR_INVALID_ARG
    assert gf(bs.BS_FP64, 0, 8, 5, A, P, I, o(il=-2), None) == bs.BS_ERR_INVALID_ARG
    assert gf(bs.BS_FP64, 0, 8, 5, A, P, I, o(t=2), None) == bs.BS_ERR_INVALID_ARG
    assert gf(bs.BS_FP64, 0, 8, 5, A, P, I, o(c=1), None) == bs.BS_ERR_UNSUPPORTED
    assert gf(bs.BS_FP64, 0, 8, 5, A, P, I, o(k=1), None) == bs.BS_ERR_UNSUPPORTED
    assert gf(bs.BS_FP64, 0, 129, 5, A, P, I, o(il=4), None) == bs.BS_ERR_UNSUPPORTED
    assert gf(bs.BS_FP64, 0, 8, 0, None, None, None, o(il=4), None) == bs.BS_OK
    assert gf(bs.BS_FP64, 0, 8, 5, A, A + 5 * 512, I, o(il=4), None) == bs.BS_ERR_INVALID_ARG
    assert gf(bs.BS_FP64, 0, 8, 5, A, P, I + 4, o(tau=0.5), None) == bs.BS_ERR_INVALID_ARG
    assert gf(bs.BS_FP64, 0, 8, 5, None, P, I, o(t=1), None) == bs.BS_ERR_INVALID_ARG
    assert gs(bs.BS_FP64, 0, 8, 2, 5, A, P, B, o(k=1), None) == bs.BS_ERR_UNSUPPORTED
    assert gs(bs.BS_FP64, 0, 8, 65537, 5, A, P, B, o(il=4), None) == bs.BS_ERR_UNSUPPORTED
    assert gs(bs.BS_FP64, 0, 8, 9, 5, A, P, A + 5 * 512, o(il=4, t=1), None) == bs.BS_ERR_INVALID_ARG
    assert gs(bs.BS_FP64, 0, 8, 9, 5, A, B + 5 * 8 * 9 * 8, B, o(il=4), None) == bs.BS_ERR_INVALID_ARG
    assert gs(bs.BS_FP64, 0, 8, 9, 0, None, None, None, o(t=1), None) == bs.BS_OK
    assert pf(bs.BS_FP64, 1, 0, 8, 5, A, I, o(t=1), None) == bs.BS_ERR_UNSUPPORTED
    assert pf(bs.BS_FP64, 1, 0, 8, 5, A, I, o(c=1), None) == bs.BS_ERR_UNSUPPORTED
    assert pf(bs.BS_FP64, 1, 0, 200, 5, A, I, o(il=4), None) == bs.BS_ERR_UNSUPPORTED
    assert pf(bs.BS_FP64, 1, 2, 8, 5, A, I, o(il=4), None) == bs.BS_ERR_UNSUPPORTED
    assert pf(bs.BS_FP64, 1, 0, 8, 5, A, A + 5 * 512, o(il=4), None) == bs.BS_ERR_INVALID_ARG
    assert ps(bs.BS_FP64, 1, 0, 8, 1, 5, A, A + 5 * 512, o(il=4), None) == bs.BS_ERR_INVALID_ARG
    assert ps(bs.BS_FP64, 1, 0, 8, 1, 5, A, B, o(k=1), None) == bs.BS_ERR_UNSUPPORTED
    assert ps(bs.BS_FP64, 1, 0, 8, 1, 0, None, None, o(il=4), None) == bs.BS_OK


def test_binding_refuses_host_tensors():
    import torch
    A = torch.zeros((2, 4, 4))
    B = torch.zeros((2, 4, 1))
    ipiv = torch.zeros((2, 4), dtype=torch.int32)
    info = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError):
        bs.bs_getrf_getrs_batched(A, B, ipiv, info)


def test_cholesky_order_limits(lib):
    """Cholesky reaches n = 256 (beyond one CTA: the cluster factor); LU stays at 128; the
    contract options and interleaved layouts stay at n <= 128."""
    import ctypes
    assert lib.bs_potrf_potrs_supported(bs.BS_FP64, bs.BS_COL_MAJOR, bs.BS_LOWER, 256, 1) == 1
    assert lib.bs_potrf_potrs_supported(bs.BS_FP32, bs.BS_ROW_MAJOR, bs.BS_UPPER, 200, 3) == 1
    assert lib.bs_potrf_potrs_supported(bs.BS_FP64, bs.BS_COL_MAJOR, bs.BS_LOWER, 257, 1) == 0
    A, B, I = FAKE, FAKE + 0x1000000, FAKE + 0x2000000
    assert lib.bs_potrf_potrs_batched(bs.BS_FP64, 1, 0, 257, 1, 5, A, B, I,
                                      None) == bs.BS_ERR_UNSUPPORTED
    assert lib.bs_potrf_batched(bs.BS_FP64, 1, 0, 300, 5, A, I, None) == bs.BS_ERR_UNSUPPORTED
    ruda = ctypes.byref(bs.Options(1.0, bs.BS_CONTRACT_RUDA, 0, 0, 0))
    assert lib.bs_potrf_potrs_batched_ex(bs.BS_FP64, 1, 0, 200, 1, 5, A, B, I, ruda,
                                         None) == bs.BS_ERR_UNSUPPORTED
    il = ctypes.byref(bs.Options(1.0, 0, 0, 4, 0))
    assert lib.bs_potrf_potrs_batched_ex(bs.BS_FP64, 1, 0, 200, 1, 8, A, B, I, il,
                                         None) == bs.BS_ERR_UNSUPPORTED


def test_host_resident_argument_errors(lib):
    """The *_host calls check everything before the first copy: chunk, workspace (null,
    misaligned, too small), host pointers, shapes; an empty batch submits nothing."""
    import ctypes
    W = 2 * (((8192 * 1024 + 255) // 256) * 256 + ((8192 * 256 + 255) // 256) * 256
             + ((8192 * 64 + 255) // 256) * 256 + ((8192 * 4 + 255) // 256) * 256)
    assert lib.bs_getrf_getrs_host_workspace(bs.BS_FP32, 16, 4, 8192) == W
    assert lib.bs_getrf_getrs_host_workspace(bs.BS_FP32, 0, 4, 8192) == 0
    assert lib.bs_potrf_potrs_host_workspace(bs.BS_FP64, 32, 1, 0) == 0
    assert lib.bs_bdsv_host_workspace(bs.BS_FP64, 32, 8, 16) > 16 * 32 * 8 * 24 * 8
    A, B, P, I, WK = FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, FAKE + 0x1000000
    f = lib.bs_getrf_getrs_batched_host
    assert f(bs.BS_FP32, 0, 16, 4, 0, None, None, None, None, None, 0, 1, None, None) == bs.BS_OK
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, WK, W, 0, None, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, None, W, 8192, None, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, WK + 16, W, 8192, None, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, WK, W - 1, 8192, None, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, None, P, I, WK, W, 8192, None, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 129, 4, 5, A, B, P, I, WK, W, 8192, None, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP32, 0, 16, -1, 5, A, B, P, I, WK, W, 8192, None, None) == bs.BS_ERR_INVALID_ARG
    g = lib.bs_potrf_potrs_batched_host
    assert g(bs.BS_FP64, 1, 0, 32, 1, 5, A, B, I, WK, 16, 8, None, None) == bs.BS_ERR_INVALID_ARG
    assert g(bs.BS_FP64, 1, 2, 32, 1, 5, A, B, I, WK, 1 << 30, 8, None, None) == bs.BS_ERR_UNSUPPORTED
    h = lib.bs_bdsv_batched_host
    assert h(bs.BS_FP64, 32, 9, 5, A, B, I, WK, 1 << 30, 8, None, None) == bs.BS_ERR_UNSUPPORTED
    assert h(bs.BS_FP64, 32, 8, 5, A, B, None, WK, 1 << 30, 8, None, None) == bs.BS_ERR_INVALID_ARG
    # a batch whose host extent (systems x bytes per system) is not representable is refused
    # before the host arrays are compared for overlap
    assert f(bs.BS_FP32, 0, 16, 4, 1 << 62, A, B, P, I, WK, W, 8192, None,
             None) == bs.BS_ERR_INVALID_ARG
    assert h(bs.BS_FP64, 32, 8, 1 << 60, A, B, I, WK, 1 << 30, 8, None,
             None) == bs.BS_ERR_INVALID_ARG


def test_aliased_operands_are_rejected(lib):
    """Operands of one call must not alias: every entry point checks the byte ranges of
    its operands (the interleaved layouts with their whole blocks) before launching."""
    import ctypes
    A = FAKE
    # LU FP32 n=16 nrhs=4 batch 5: A takes 5 KB; B placed inside it, then just after it
    assert lib.bs_getrf_getrs_batched(bs.BS_FP32, 0, 16, 4, 5, A, A + 4096, A + 0x100000,
                                      A + 0x200000, None) == bs.BS_ERR_INVALID_ARG
    assert lib.bs_getrf_getrs_batched(bs.BS_FP32, 0, 16, 4, 5, A, A + 0x100000, A + 0x100000 + 1264,
                                      A + 0x200000, None) == bs.BS_ERR_INVALID_ARG
    assert lib.bs_getrf_getrs_batched(bs.BS_FP32, 0, 16, 4, 5, A, A + 0x100000, A + 0x200000,
                                      A + 0x200000 + 304, None) == bs.BS_ERR_INVALID_ARG
    assert lib.bs_potrf_potrs_batched(bs.BS_FP64, 1, 0, 32, 1, 5, A, A + 40960 - 16,
                                      A + 0x100000, None) == bs.BS_ERR_INVALID_ARG
    assert lib.bs_bdsv_batched(bs.BS_FP64, 32, 8, 2, A, A + 0x100000, A + 0x100000 + 528,
                               None) == bs.BS_ERR_INVALID_ARG
    assert lib.bs_getrf_batched(bs.BS_FP64, 1, 8, 3, A, A + 8 * 8 * 8 * 2, A + 0x100000,
                                None) == bs.BS_ERR_INVALID_ARG
    assert lib.bs_potrf_batched(bs.BS_FP64, 1, 0, 8, 3, A, A + 512, None) == bs.BS_ERR_INVALID_ARG
    assert lib.bs_bdsv_factor_batched(bs.BS_FP64, 4, 2, 3, A, A + 16, None) == bs.BS_ERR_INVALID_ARG
    # interleaved: 5 systems in blocks of 4 hold 8 systems' room (8 KB for FP64 n=8)
    o = ctypes.byref(bs.Options(1.0, 0, 0, 4, 0))
    assert lib.bs_getrf_getrs_batched_ex(bs.BS_FP64, 0, 8, 1, 5, A, A + 5 * 512, A + 0x100000,
                                         A + 0x200000, o, None) == bs.BS_ERR_INVALID_ARG
    # host arrays of the host-resident call
    W = lib.bs_getrf_getrs_host_workspace(bs.BS_FP32, 16, 4, 8)
    assert lib.bs_getrf_getrs_batched_host(bs.BS_FP32, 0, 16, 4, 5, A, A + 1024, A + 0x100000,
                                           A + 0x200000, A + 0x1000000, W, 8, None,
                                           None) == bs.BS_ERR_INVALID_ARG


def _cpu(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a))


def _refused_as_host(fn, *args, **kw):
    """The operand checks pass; the call then stops at the device check of the first
    pointer (these are CPU tensors), before anything reaches the library."""
    with pytest.raises(ValueError, match="device tensors"):
        fn(*args, **kw)


def test_binding_operand_checks_accept_the_workloads():
    """Every workload's operands, shaped as the tests and the benchmark pass them, get
    through the binding's dtype / shape checks of every wrapper."""
    import torch
    from gen import workloads as W
    for name, w in W.WORKLOADS.items():
        d = W.make(name, 37)
        if w.op == "bdsv":
            S, X = _cpu(d["strips"]), _cpu(d["x"])
            info = torch.zeros(37, dtype=torch.int32)
            _refused_as_host(bs.bs_bdsv_batched, S, X, info)
            _refused_as_host(bs.bs_bdsv_factor_batched, S, info)
            _refused_as_host(bs.bs_bdsv_solve_batched, S, X)
            _refused_as_host(bs.bs_bdmv_batched, S, X, X.clone())
            _refused_as_host(bs.bs_bdmv2_batched, S, X, X.clone(), X.clone())
            continue
        A, B = _cpu(d["A"]), _cpu(d["B"])
        n = A.shape[1]
        ipiv = torch.zeros((37, n), dtype=torch.int32)
        info = torch.zeros(37, dtype=torch.int32)
        if w.op == "getrf_getrs":
            _refused_as_host(bs.bs_getrf_getrs_batched, A, B, ipiv, info, w.layout)
            _refused_as_host(bs.bs_getrf_batched, A, ipiv, info, w.layout)
            _refused_as_host(bs.bs_getrs_batched, A, ipiv, B, w.layout)
            _refused_as_host(bs.bs_getrf_getrs_batched_ex, A, B, ipiv, info, w.layout, 0.5)
            for wd in (4, 32, 40):   # interleaved: flat operands holding whole blocks
                Ai, Bi = _cpu(W.interleave(d["A"], wd)), _cpu(W.interleave(d["B"], wd))
                ip = torch.zeros(Ai.numel() // n, dtype=torch.int32)
                _refused_as_host(bs.bs_getrf_getrs_batched_ex, Ai, Bi, ip, info, w.layout,
                                 interleave=wd, shape=(37, n, w.nrhs))
        else:
            _refused_as_host(bs.bs_potrf_potrs_batched, A, B, info, w.layout)
            _refused_as_host(bs.bs_potrf_batched, A, info, w.layout)
            _refused_as_host(bs.bs_potrs_batched, A, B, w.layout)
            Ai, Bi = _cpu(W.interleave(d["A"], 37)), _cpu(W.interleave(d["B"], 37))
            _refused_as_host(bs.bs_potrf_potrs_batched_ex, Ai, Bi, info, w.layout,
                             interleave=37, shape=(37, n, w.nrhs))


def test_binding_operand_checks_reject_mismatches():
    """A tensor of another dtype or size than the call's shape implies is refused with a
    TypeError / ValueError naming the operand, before any pointer reaches the library
    (which would otherwise read it as the expected type and size)."""
    import torch
    A = torch.zeros((5, 16, 16))
    B = torch.zeros((5, 16, 4))
    ipiv = torch.zeros((5, 16), dtype=torch.int32)
    info = torch.zeros(5, dtype=torch.int32)
    f = bs.bs_getrf_getrs_batched
    with pytest.raises(TypeError, match="B: dtype"):
        f(A, B.double(), ipiv, info)
    with pytest.raises(TypeError, match="ipiv: dtype"):
        f(A, B, ipiv.long(), info)
    with pytest.raises(TypeError, match="info: dtype"):
        f(A, B, ipiv, info.float())
    with pytest.raises(ValueError, match="info: 4 elements"):
        f(A, B, ipiv, info[:4])
    with pytest.raises(ValueError, match="ipiv: 75 elements"):
        f(A, B, ipiv[:, :15].contiguous(), info)
    with pytest.raises(ValueError, match="A: shape"):
        f(A[:, :, :15].contiguous(), B, ipiv, info)
    with pytest.raises(ValueError, match="B: shape"):
        f(A, torch.zeros((4, 16, 4)), ipiv, info)
    with pytest.raises(ValueError, match="B: shape"):          # column-major B is (batch, nrhs, n)
        f(A, B, ipiv, info, COL)
    with pytest.raises(TypeError, match="unsupported dtype"):
        f(A.half(), B.half(), ipiv, info)
    with pytest.raises(ValueError, match="B: shape"):
        bs.bs_potrs_batched(A.double(), torch.zeros((5, 16), dtype=torch.float64))
    S = torch.zeros((3, 32, 8, 24), dtype=torch.float64)
    X = torch.zeros((3, 34 * 8), dtype=torch.float64)
    binfo = torch.zeros(3, dtype=torch.int32)
    with pytest.raises(ValueError, match="strips: shape"):
        bs.bs_bdsv_batched(S[..., :16].contiguous(), X, binfo)
    with pytest.raises(ValueError, match="x_padded: 264 elements"):
        bs.bs_bdsv_batched(S, X[:, :88].contiguous(), binfo)
    with pytest.raises(TypeError, match="y_padded: dtype"):
        bs.bs_bdmv_batched(S, X, X.float())
    # interleaved: ipiv and B hold whole blocks (5 systems in blocks of 4: 8 systems' room)
    Ai, Bi = torch.zeros(8 * 256), torch.zeros(8 * 64)
    with pytest.raises(ValueError, match="ipiv: 80 elements"):
        bs.bs_getrf_getrs_batched_ex(Ai, Bi, torch.zeros(80, dtype=torch.int32), info,
                                     interleave=4, shape=(5, 16, 4))
    with pytest.raises(ValueError, match="B: 320 elements"):
        bs.bs_getrf_getrs_batched_ex(Ai, Bi[:320].contiguous(),
                                     torch.zeros(128, dtype=torch.int32), info,
                                     interleave=4, shape=(5, 16, 4))
    # host-resident calls check the same before planning anything
    with pytest.raises(TypeError, match="B: dtype"):
        bs.bs_getrf_getrs_batched_host(A, B.double(), ipiv, info)
    with pytest.raises(ValueError, match="info: 4 elements"):
        bs.bs_potrf_potrs_batched_host(A.double(), torch.zeros((5, 4, 16), dtype=torch.float64),
                                       info[:4], COL)
    with pytest.raises(ValueError, match="x_padded"):
        bs.bs_bdsv_batched_host(S, X[:2].contiguous(), binfo)


def test_huge_chunks_do_not_wrap_the_workspace_size(lib):
    """A chunk whose slots would not fit any memory makes the workspace queries return 0
    (no wrapped-around small size), and a host call with such a chunk is refused before
    any copy (the workspace it needs exceeds any that can be passed)."""
    huge = 2 ** 62
    assert lib.bs_getrf_getrs_host_workspace(bs.BS_FP32, 16, 4, huge) == 0
    assert lib.bs_potrf_potrs_host_workspace(bs.BS_FP64, 32, 1, huge) == 0
    assert lib.bs_bdsv_host_workspace(bs.BS_FP64, 32, 8, huge) == 0
    assert lib.bs_getrf_getrs_host_workspace(bs.BS_FP32, 16, 4, 2 ** 40) > 2 ** 40 * 1348
    A, B, P, I, WK = FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, FAKE + 0x1000000
    for chunk in (huge, 2 ** 63 - 1):
        assert lib.bs_getrf_getrs_batched_host(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, WK, 4096,
                                               chunk, None, None) == bs.BS_ERR_INVALID_ARG
        assert lib.bs_potrf_potrs_batched_host(bs.BS_FP64, 1, 0, 32, 1, 5, A, B, I, WK, 4096,
                                               chunk, None, None) == bs.BS_ERR_INVALID_ARG
        assert lib.bs_bdsv_batched_host(bs.BS_FP64, 32, 8, 5, A, B, I, WK, 4096, chunk, None,
                                        None) == bs.BS_ERR_INVALID_ARG
