"""The options of the _ex calls in combination, and the split calls with options, against
the CPU oracle bit for bit through the C ABI.

TDLS's row-major reading (the factor of the stored array read column-major, then the
mirror solve) on the interleaved batched layouts, with a pivot threshold and with RUDA's
max-abs scaling; getrf/getrs and potrf/potrs alone on the interleaved layouts, getrf
under a threshold and under the row-major reading, getrs with the mirror solve. LU
comparisons skip the systems where the oracle met a near tie in the pivot search (the
same rule as every other LU parity test); Cholesky has no pivot search and compares
every system that factored.
"""
import os

import numpy as np
import pytest
import torch

import dense_linear_solvers_gb300 as bs
import oracle
from gen.workloads import COL_MAJOR, ROW_MAJOR, deinterleave, interleave, to_storage
from tests import parity

pytestmark = pytest.mark.gpu
NT = os.cpu_count() or 1
SENT = parity.SENTINEL


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bs.lib()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def _lu_case(rng, dtype, batch, n, nrhs, layout):
    Al = rng.uniform(-1, 1, (batch, n, n)).astype(dtype)
    Al[1] *= dtype(1e-3)                     # magnitudes away from 1 for the scaling
    Al[2, :, n // 2] = 0                     # a zero column of A (a zero row of S)
    Al[3, n // 2, :] = 0                     # a zero row of A (a zero column of S)
    Bl = rng.standard_normal((batch, n, nrhs)).astype(dtype)
    return to_storage(Al, layout), to_storage(Bl, layout)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_row_major_reading_interleaved_scaled(dtype):
    """transposed_factor with interleave W in {4, 32, batch, batch + 3}, with the threshold
    and with the scaling, orders over the register sizes and the one-CTA sizes, and
    right-hand-side counts past the 8 a solve pass takes."""
    rng = np.random.default_rng(2121)
    batch = 19
    for n in (1, 3, 8, 16, 31, 33, 64, 128):
        for w, tau, scale in ((4, 1.0, 0), (32, 0.5, 0), (batch, 1.0, 1), (batch + 3, 0.5, 1),
                              (1, 1.0, 1)):
            nrhs = int(rng.choice([1, 3, 8, 11]))
            A, B = _lu_case(rng, dtype, batch, n, nrhs, ROW_MAJOR)
            Af, Bf = interleave(A, w), interleave(B, w)
            So, Xo, ipo, info_o, tie = oracle.getrf_getrs_mirror_il(
                Af, Bf, n, nrhs, batch, w, ROW_MAJOR, tau=tau, scale=scale, nthreads=NT)
            tA, tB = _dev(Af), _dev(Bf)
            ipiv = torch.full((Af.size // n,), SENT, dtype=torch.int32, device="cuda")
            info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
            if w == 1:   # the plain layout: the binding takes the batched shapes
                bs.bs_getrf_getrs_batched_ex(tA.view(A.shape), tB.view(B.shape),
                                             ipiv.view(batch, n), info, ROW_MAJOR, tau,
                                             transposed_factor=1, scaling=scale)
            else:
                bs.bs_getrf_getrs_batched_ex(tA, tB, ipiv, info, ROW_MAJOR, tau,
                                             transposed_factor=1, interleave=w,
                                             shape=(batch, n, nrhs), scaling=scale)
            Ag, Bg, ipg, infg = _host(tA), _host(tB), _host(ipiv), _host(info)
            clean = tie < 0
            key = (n, w, tau, scale)
            assert clean.sum() >= batch - 3, key
            assert np.array_equal(infg[clean], info_o[clean]), key
            if n > 1:
                assert infg[2] > 0 and infg[3] > 0, key
            for got, ref, shape in ((Ag, So, (n, n)), (Bg, Xo, B.shape[1:]), (ipg, ipo, (n,))):
                g2, r2 = deinterleave(got, batch, w, shape), deinterleave(ref, batch, w, shape)
                assert np.array_equal(g2[clean], r2[clean]), key
            Xg = deinterleave(Bg, batch, w, B.shape[1:])
            assert np.all(Xg[infg != 0] == 0), key
            # the slots of the last block past the batch are neither read nor written
            pads = np.isnan(interleave(np.zeros((batch,) + B.shape[1:]), w))
            assert np.all(np.isnan(Bg[pads])), key


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_split_lu_interleaved(dtype, layout):
    """getrf alone on an interleaved layout = the oracle's interleaved getrf; getrs alone
    from the oracle's factor = the oracle's getrs; the two in a row = the fused call."""
    rng = np.random.default_rng(2222 + layout)
    batch = 23
    for n in (2, 16, 32, 40, 128):
        for w in (3, 32, batch + 1):
            nrhs = int(rng.choice([1, 4, 9]))
            A, B = _lu_case(rng, dtype, batch, n, nrhs, layout)
            Af, Bf = interleave(A, w), interleave(B, w)
            Fo, ipo, info_o, tie = oracle.getrf_il(Af, n, batch, w, layout, nthreads=NT)
            tA = _dev(Af)
            ipiv = torch.full((Af.size // n,), SENT, dtype=torch.int32, device="cuda")
            info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
            bs.bs_getrf_batched_ex(tA, ipiv, info, layout, interleave=w, shape=(batch, n))
            Fg, ipg, infg = _host(tA), _host(ipiv), _host(info)
            clean = tie < 0
            assert clean.sum() >= batch - 3 and np.array_equal(infg[clean], info_o[clean])
            for got, ref, shape in ((Fg, Fo, (n, n)), (ipg, ipo, (n,))):
                g2, r2 = deinterleave(got, batch, w, shape), deinterleave(ref, batch, w, shape)
                assert np.array_equal(g2[clean], r2[clean]), (n, w)
            # the solve from the oracle's factor (every system that factored)
            Xo = oracle.getrs_il(Fo, ipo, Bf, n, nrhs, batch, w, layout, nthreads=NT)
            tB = _dev(Bf)
            bs.bs_getrs_batched_ex(_dev(Fo), _dev(ipo), tB, layout, interleave=w,
                                   shape=(batch, n, nrhs))
            ok = info_o == 0
            Xg = _host(tB)
            shape = B.shape[1:]
            assert np.array_equal(deinterleave(Xg, batch, w, shape)[ok],
                                  deinterleave(Xo, batch, w, shape)[ok]), (n, w)
            pads = np.isnan(interleave(np.zeros((batch,) + shape), w))
            assert np.all(np.isnan(Xg[pads]))
            # factor then solve on the device = the fused interleaved call (nrhs <= 8)
            if nrhs > 8:
                continue
            tA2, tB2 = _dev(Af), _dev(Bf)
            ip2 = torch.full((Af.size // n,), SENT, dtype=torch.int32, device="cuda")
            in2 = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
            bs.bs_getrf_getrs_batched_ex(tA2, tB2, ip2, in2, layout, interleave=w,
                                         shape=(batch, n, nrhs))
            tB3 = _dev(Bf)
            bs.bs_getrs_batched_ex(tA, ipiv, tB3, layout, interleave=w, shape=(batch, n, nrhs))
            okg = infg == 0
            assert np.array_equal(_host(tA2), Fg, equal_nan=True)
            assert np.array_equal(_host(ip2), ipg)
            assert np.array_equal(deinterleave(_host(tB3), batch, w, shape)[okg],
                                  deinterleave(_host(tB2), batch, w, shape)[okg]), (n, w)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_split_lu_threshold_and_row_major_reading(dtype):
    """getrf alone under a threshold = the fused call's factor; under the row-major reading
    = the oracle's mirror factor; getrs alone with the mirror solve from the oracle's
    mirror factor = the oracle's X."""
    rng = np.random.default_rng(2323)
    batch = 17
    for n in (1, 5, 16, 32, 33, 100):
        nrhs = int(rng.choice([1, 2, 8, 13]))
        for layout in (ROW_MAJOR, COL_MAJOR):
            A, B = _lu_case(rng, dtype, batch, n, nrhs, layout)
            Fo, Xo, ipo, info_o, tie = oracle.getrf_getrs_ex(A, B, layout, tau=0.5, nthreads=NT)
            tA = _dev(A)
            ipiv = torch.full((batch, n), SENT, dtype=torch.int32, device="cuda")
            info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
            bs.bs_getrf_batched_ex(tA, ipiv, info, layout, pivot_threshold=0.5)
            clean = tie < 0
            assert clean.sum() >= batch - 3
            assert np.array_equal(_host(tA)[clean], Fo[clean]), (n, layout)
            assert np.array_equal(_host(ipiv)[clean], ipo[clean])
            assert np.array_equal(_host(info)[clean], info_o[clean])
        A, B = _lu_case(rng, dtype, batch, n, nrhs, ROW_MAJOR)
        So, Xo, ipo, info_o, tie = oracle.getrf_getrs_mirror(A, B, ROW_MAJOR, nthreads=NT)
        tA = _dev(A)
        ipiv = torch.full((batch, n), SENT, dtype=torch.int32, device="cuda")
        info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
        bs.bs_getrf_batched_ex(tA, ipiv, info, ROW_MAJOR, transposed_factor=1)
        clean = tie < 0
        assert np.array_equal(_host(tA)[clean], So[clean]), n
        assert np.array_equal(_host(ipiv)[clean], ipo[clean])
        assert np.array_equal(_host(info)[clean], info_o[clean])
        tB = _dev(B)
        bs.bs_getrs_batched_ex(_dev(So), _dev(ipo), tB, ROW_MAJOR, transposed_factor=1)
        ok = info_o == 0
        assert np.array_equal(_host(tB)[ok], Xo[ok]), n


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
@pytest.mark.parametrize("fill", [bs.BS_LOWER, bs.BS_UPPER])
def test_split_cholesky_interleaved(dtype, layout, fill):
    """potrf alone on an interleaved layout = the oracle's (the other triangle untouched,
    NaN there); potrs alone from the oracle's factor = the oracle's X; the two in a row =
    the fused interleaved call."""
    rng = np.random.default_rng(2424 + 2 * layout + fill)
    batch = 21
    for n in (1, 4, 31, 32, 33, 64, 128):
        for w in (2, 32, batch + 2):
            nrhs = int(rng.choice([1, 3, 8, 10]))
            G = rng.standard_normal((batch, n, n))
            Al = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dtype)
            Al[batch // 2, n - 1, n - 1] = -1.0
            iu = np.triu_indices(n, 1) if fill == bs.BS_LOWER else np.tril_indices(n, -1)
            Al[:, iu[0], iu[1]] = np.nan
            A = to_storage(Al, layout)
            B = to_storage(rng.standard_normal((batch, n, nrhs)).astype(dtype), layout)
            Af, Bf = interleave(A, w), interleave(B, w)
            Lo, info_o = oracle.potrf_il(Af, n, batch, w, layout, fill, nthreads=NT)
            tA = _dev(Af)
            info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
            bs.bs_potrf_batched_ex(tA, info, layout, fill, interleave=w, shape=(batch, n))
            Lg = _host(tA)
            assert np.array_equal(_host(info), info_o) and info_o[batch // 2] == n, (n, w)
            ok = info_o == 0
            g2, r2 = deinterleave(Lg, batch, w, (n, n)), deinterleave(Lo, batch, w, (n, n))
            assert np.array_equal(g2[ok], r2[ok], equal_nan=True), (n, w)
            if n > 1:
                assert np.all(np.isnan(g2[:, iu[0], iu[1]]) if layout == ROW_MAJOR
                              else np.isnan(np.swapaxes(g2, 1, 2)[:, iu[0], iu[1]]))
            Xo = oracle.potrs_il(Lo, Bf, n, nrhs, batch, w, layout, fill, nthreads=NT)
            tB = _dev(Bf)
            bs.bs_potrs_batched_ex(_dev(Lo), tB, layout, fill, interleave=w,
                                   shape=(batch, n, nrhs))
            shape = B.shape[1:]
            Xg = _host(tB)
            assert np.array_equal(deinterleave(Xg, batch, w, shape)[ok],
                                  deinterleave(Xo, batch, w, shape)[ok]), (n, w)
            pads = np.isnan(interleave(np.zeros((batch,) + shape), w))
            assert np.all(np.isnan(Xg[pads]))
            if nrhs > 8:   # the fused interleaved call takes 8 right-hand sides at most
                continue
            tA2, tB2 = _dev(Af), _dev(Bf)
            in2 = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
            bs.bs_potrf_potrs_batched_ex(tA2, tB2, in2, layout, fill, interleave=w,
                                         shape=(batch, n, nrhs))
            tB3 = _dev(Bf)
            bs.bs_potrs_batched_ex(tA, tB3, layout, fill, interleave=w, shape=(batch, n, nrhs))
            assert np.array_equal(deinterleave(_host(tA2), batch, w, (n, n))[ok], g2[ok],
                                  equal_nan=True)
            assert np.array_equal(deinterleave(_host(tB3), batch, w, shape)[ok],
                                  deinterleave(_host(tB2), batch, w, shape)[ok]), (n, w)


def test_split_options_refused():
    """The options that span the factor and the solve stay with the fused calls; Cholesky
    takes no LU option; interleaved Cholesky stays at n <= 128."""
    A = torch.zeros((4, 8, 8), dtype=torch.float64, device="cuda")
    ipiv = torch.zeros((4, 8), dtype=torch.int32, device="cuda")
    info = torch.zeros(4, dtype=torch.int32, device="cuda")
    B = torch.zeros((4, 8, 2), dtype=torch.float64, device="cuda")
    cases = [
        lambda: bs.bs_getrf_batched_ex(A, ipiv, info, status_contract=bs.BS_CONTRACT_RUDA),
        lambda: bs.bs_getrf_batched_ex(A, ipiv, info, scaling=1),
        lambda: bs.bs_getrs_batched_ex(A, ipiv, B, scaling=1),
        lambda: bs.bs_potrf_batched_ex(A, info, transposed_factor=1),
        lambda: bs.bs_potrf_batched_ex(A, info, status_contract=bs.BS_CONTRACT_RUDA),
    ]
    for c in cases:
        with pytest.raises(bs.BsolveError) as e:
            c()
        assert e.value.status == bs.BS_ERR_UNSUPPORTED
    Ab = torch.zeros(4 * 160 * 160, dtype=torch.float64, device="cuda")
    with pytest.raises(bs.BsolveError) as e:
        bs.bs_potrf_batched_ex(Ab, info, interleave=4, shape=(4, 160))
    assert e.value.status == bs.BS_ERR_UNSUPPORTED
