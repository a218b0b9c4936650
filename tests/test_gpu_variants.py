"""Contract variants of the fused calls (TDLS threshold pivoting, RUDA status contract):
the CUDA path through the C ABI against the CPU oracle, bit for bit.

Threshold pivoting over the orders 1..128 with both layouts and dtypes (compared on the
systems where the oracle met no near tie, pivot choice included); the RUDA contract on
constructed systems for every status code (-1 non-finite input, -2 non-symmetric,
k > 0 failing pivot or minor, -3 overflow), both fills for Cholesky.
"""
import os

import numpy as np
import pytest
import torch

import dense_linear_solvers_gb300 as bs
import oracle
from gen.workloads import COL_MAJOR, ROW_MAJOR, to_storage
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


def gpu_lu_ex(A, B, layout, tau, contract):
    tA, tB = _dev(A), _dev(B)
    batch, n = A.shape[0], A.shape[1]
    ipiv = torch.full((batch, n), SENT, dtype=torch.int32, device="cuda")
    info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
    bs.bs_getrf_getrs_batched_ex(tA, tB, ipiv, info, layout, tau, contract)
    return _host(tA), _host(tB), _host(ipiv), _host(info)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_threshold_pivoting(dtype, layout):
    rng = np.random.default_rng(1212 + layout)
    for n in list(range(1, 40)) + [64, 100, 128]:
        for tau in (0.3, 0.8):
            nrhs = int(rng.integers(1, 9))
            Al = rng.standard_normal((17, n, n)).astype(dtype)
            if n > 1:
                Al[3, :, n // 2] = 0
            A = to_storage(Al, layout)
            B = to_storage(rng.standard_normal((17, n, nrhs)).astype(dtype), layout)
            LUo, Xo, ipo, info_o, tie = oracle.getrf_getrs_ex(A, B, layout, tau=tau, nthreads=NT)
            LUg, Xg, ipg, infg = gpu_lu_ex(A, B, layout, tau, bs.BS_CONTRACT_DEFAULT)
            clean = tie < 0
            assert np.array_equal(infg[clean], info_o[clean]), (n, tau)
            assert np.array_equal(ipg[clean], ipo[clean]), (n, tau)
            assert np.array_equal(LUg[clean], LUo[clean]) and np.array_equal(Xg[clean], Xo[clean])
            assert np.all(Xg[infg != 0] == 0)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_ruda_status_lu(dtype, layout):
    rng = np.random.default_rng(1313 + layout)
    big = np.finfo(dtype).max
    for n in (2, 4, 16, 40, 128):
        Al = rng.standard_normal((6, n, n)).astype(dtype) + 3 * np.eye(n, dtype=dtype)
        Bl = rng.standard_normal((6, n, 2)).astype(dtype)
        Al[0, n - 1, 0] = np.nan
        Bl[1, 0, 1] = -np.inf
        Al[2, :, n - 1] = 0
        Al[3] = np.eye(n, dtype=dtype)
        Al[3, 0, 0] = np.finfo(dtype).tiny * 2
        Bl[3, 0, 0] = big / 2
        A, B = to_storage(Al, layout), to_storage(Bl, layout)
        LUo, Xo, ipo, info_o, tie = oracle.getrf_getrs_ex(A, B, layout, ruda=1)
        LUg, Xg, ipg, infg = gpu_lu_ex(A, B, layout, 1.0, bs.BS_CONTRACT_RUDA)
        assert list(info_o) == [-1, -1, n, -3, 0, 0], info_o
        assert np.array_equal(infg, info_o)
        assert np.array_equal(ipg, ipo) and np.array_equal(LUg, LUo) and np.array_equal(Xg, Xo)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_ruda_status_cholesky(dtype, layout):
    rng = np.random.default_rng(1414 + layout)
    for n in (1, 3, 16, 33, 128):
        G = rng.standard_normal((7, n, n))
        Al = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dtype)
        Bl = rng.standard_normal((7, n, 3)).astype(dtype)
        Al[0, n - 1, n - 1] = np.nan
        Bl[1, n - 1, 2] = np.inf
        if n > 1:
            Al[2, n - 1, 0] = np.nextafter(Al[2, n - 1, 0], dtype(np.inf))
        Al[3, n - 1, n - 1] = -1.0
        Al[4] = np.diag(np.full(n, np.finfo(dtype).tiny * 4)).astype(dtype)
        Bl[4] = np.finfo(dtype).max / 8
        A, B = to_storage(Al, layout), to_storage(Bl, layout)
        for fill in (bs.BS_LOWER, bs.BS_UPPER):
            Lo, Xo, info_o = oracle.potrf_potrs_ex(A, B, layout, fill=fill, ruda=1)
            tA, tB = _dev(A), _dev(B)
            info = torch.full((7,), SENT, dtype=torch.int32, device="cuda")
            bs.bs_potrf_potrs_batched_ex(tA, tB, info, layout, fill, bs.BS_CONTRACT_RUDA)
            want = [-1, -1, -2 if n > 1 else 0, n, -3, 0, 0]
            assert list(info_o) == want, (n, fill, info_o)
            assert np.array_equal(_host(info), info_o)
            assert np.array_equal(_host(tA), Lo, equal_nan=True)
            assert np.array_equal(_host(tB), Xo)


def gpu_lu_mirror(A, B, layout, tau):
    tA, tB = _dev(A), _dev(B)
    batch, n = A.shape[0], A.shape[1]
    ipiv = torch.full((batch, n), SENT, dtype=torch.int32, device="cuda")
    info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
    bs.bs_getrf_getrs_batched_ex(tA, tB, ipiv, info, layout, tau, bs.BS_CONTRACT_DEFAULT,
                                 transposed_factor=1)
    return _host(tA), _host(tB), _host(ipiv), _host(info)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("tau", [1.0, 0.5])
def test_transposed_factor_row_major(dtype, tau):
    """TDLS's row-major reading: factor of A^T in the stored array, mirror solve; every
    register tier, the shared-memory tiers, ragged right-hand-side chunks, singular
    systems."""
    rng = np.random.default_rng(1414 + int(tau * 10))
    orders = list(range(1, 34)) + [40, 64, 65, 100, 128]
    for n in orders:
        nrhs = int(rng.choice([1, 2, 3, 4, 7, 8, 9, 20]))
        Al = rng.standard_normal((23, n, n)).astype(dtype)
        Al[5, n // 2, :] = 0           # a zero row of A: a zero column of S
        if n > 1:
            Al[7, :, 0] = Al[7, :, n - 1]   # equal columns of A: a singular S as well
        Bl = rng.standard_normal((23, n, nrhs)).astype(dtype)
        So, Xo, ipo, info_o, tie = oracle.getrf_getrs_mirror(Al, Bl, ROW_MAJOR, tau=tau,
                                                              nthreads=NT)
        Sg, Xg, ipg, infg = gpu_lu_mirror(Al, Bl, ROW_MAJOR, tau)
        clean = tie < 0
        assert clean.sum() >= 20, n
        assert np.array_equal(infg[clean], info_o[clean]), (n, nrhs)
        assert np.array_equal(ipg[clean], ipo[clean]), (n, nrhs)
        assert np.array_equal(Sg[clean], So[clean]), (n, nrhs)
        assert np.array_equal(Xg[clean], Xo[clean]), (n, nrhs)
        assert infg[5] > 0 and np.all(Xg[infg != 0] == 0)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_transposed_factor_col_major_is_plain(dtype):
    """Under column-major storage S = A: the option runs the plain call, bit for bit."""
    rng = np.random.default_rng(1515)
    for n in (3, 16, 32, 50):
        A = to_storage(rng.standard_normal((9, n, n)).astype(dtype), COL_MAJOR)
        B = to_storage(rng.standard_normal((9, n, 4)).astype(dtype), COL_MAJOR)
        r1 = gpu_lu_mirror(A, B, COL_MAJOR, 1.0)
        r2 = gpu_lu_ex(A, B, COL_MAJOR, 1.0, bs.BS_CONTRACT_DEFAULT)
        assert all(np.array_equal(x, y) for x, y in zip(r1, r2))


# ------------------------------------------------------------ interleaved batched layouts
def _il_case(rng, dtype, batch, n, nrhs, layout, spd=False):
    if spd:
        G = rng.standard_normal((batch, n, n))
        Al = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dtype)
        Al[batch // 2, n - 1, n - 1] = -1.0          # a failing minor
    else:
        Al = rng.standard_normal((batch, n, n)).astype(dtype)
        Al[batch // 2, :, n // 2] = 0                # a singular system
    Bl = rng.standard_normal((batch, n, nrhs)).astype(dtype)
    return to_storage(Al, layout), to_storage(Bl, layout)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_interleaved_lu(dtype, layout):
    """AoSoA (blocks of 2, 3, 16 and 32, the last block ragged), SoA (W = batch) and SoA
    with spare capacity, every tier of the register kernel and the one-CTA kernel,
    against the oracle bit for bit; the slots past the batch are never written. Blocks of
    16 and 32 take the staged path for whole groups of sixteen systems and the
    element-wise one for the ragged rest."""
    from gen.workloads import deinterleave, interleave
    rng = np.random.default_rng(1616 + layout)
    batch = 45
    for n in (1, 2, 3, 5, 8, 13, 16, 17, 31, 32, 33, 40, 64, 65, 128):
        for w in (2, 3, 16, 32, batch, batch + 5):
            nrhs = int(rng.integers(1, 9))
            A, B = _il_case(rng, dtype, batch, n, nrhs, layout)
            Af, Bf = interleave(A, w), interleave(B, w)
            So, Xo, ipo, info_o, tie = oracle.getrf_getrs_il(Af, Bf, n, nrhs, batch, w, layout,
                                                             nthreads=NT)
            tA, tB = _dev(Af), _dev(Bf)
            ipiv = torch.full((Af.size // n,), SENT, dtype=torch.int32, device="cuda")
            info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
            bs.bs_getrf_getrs_batched_ex(tA, tB, ipiv, info, layout, interleave=w,
                                         shape=(batch, n, nrhs))
            Ag, Bg, ipg, infg = _host(tA), _host(tB), _host(ipiv), _host(info)
            clean = tie < 0
            assert clean.sum() >= batch - 3, (n, w)
            for got, ref, shape in ((Ag, So, A.shape[1:]), (Bg, Xo, B.shape[1:])):
                g2 = deinterleave(got, batch, w, shape)
                r2 = deinterleave(ref, batch, w, shape)
                assert np.array_equal(g2[clean], r2[clean]), (n, w)
                assert np.all(np.isnan(got[np.isnan(interleave(np.zeros((batch,) + shape), w))]))
            pg = deinterleave(ipg, batch, w, (n,))
            assert np.array_equal(pg[clean], deinterleave(ipo, batch, w, (n,))[clean]), (n, w)
            pads = np.isnan(interleave(np.zeros((batch, n)), w))
            assert np.all(ipg[:pads.size][pads] == SENT)
            assert np.array_equal(infg[clean], info_o[clean]) and infg[batch // 2] > 0


@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
@pytest.mark.parametrize("nrhs", [0, 1, 2, 3, 4, 8])
def test_interleaved_lu_staged_blocks(layout, nrhs):
    """FP32 n = 16 on AoSoA blocks of 16, 32 and 48 and on SoA: whole groups of sixteen
    systems go through shared memory (the staged launch), the ragged rest element by
    element (a second launch); every right-hand-side tier and getrf alone, against the
    oracle bit for bit."""
    from gen.workloads import deinterleave, interleave
    rng = np.random.default_rng(1717 + 10 * nrhs + layout)
    n, batch = 16, 16 * 6 + 5
    for w in (16, 32, 48, batch):
        A, B = _il_case(rng, np.float32, batch, n, max(nrhs, 1), layout)
        A[7] = rng.integers(-2, 3, (n, n)).astype(np.float32)     # exact ties
        Af, Bf = interleave(A, w), interleave(B, w)
        tA = _dev(Af)
        ipiv = torch.full((Af.size // n,), SENT, dtype=torch.int32, device="cuda")
        info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
        if nrhs == 0:
            Fo, ipo, info_o, tie = oracle.getrf_il(Af, n, batch, w, layout, nthreads=NT)
            bs.bs_getrf_batched_ex(tA, ipiv, info, layout, interleave=w, shape=(batch, n))
        else:
            Fo, Xo, ipo, info_o, tie = oracle.getrf_getrs_il(Af, Bf, n, nrhs, batch, w, layout,
                                                             nthreads=NT)
            tB = _dev(Bf)
            bs.bs_getrf_getrs_batched_ex(tA, tB, ipiv, info, layout, interleave=w,
                                         shape=(batch, n, nrhs))
            Xg = _host(tB)
            assert np.array_equal(deinterleave(Xg, batch, w, B.shape[1:])[tie < 0],
                                  deinterleave(Xo, batch, w, B.shape[1:])[tie < 0]), w
        clean = tie < 0
        assert clean.sum() >= batch - 3, w
        Fg, ipg, infg = _host(tA), _host(ipiv), _host(info)
        assert np.array_equal(deinterleave(Fg, batch, w, (n, n))[clean],
                              deinterleave(Fo, batch, w, (n, n))[clean]), w
        assert np.array_equal(deinterleave(ipg, batch, w, (n,))[clean],
                              deinterleave(ipo, batch, w, (n,))[clean]), w
        assert np.array_equal(infg[clean], info_o[clean]) and infg[batch // 2] > 0
        pads = np.isnan(interleave(np.zeros((batch, n)), w))
        assert np.all(ipg[:pads.size][pads] == SENT)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
@pytest.mark.parametrize("fill", [bs.BS_LOWER, bs.BS_UPPER])
def test_interleaved_cholesky(dtype, layout, fill):
    from gen.workloads import deinterleave, interleave
    rng = np.random.default_rng(1717 + 2 * layout + fill)
    batch = 37
    for n in (1, 2, 4, 7, 16, 31, 32, 33, 64, 100):
        for w in (2, 16, 32, batch, batch + 3):
            nrhs = int(rng.integers(1, 9))
            A, B = _il_case(rng, dtype, batch, n, nrhs, layout, spd=True)
            Af, Bf = interleave(A, w), interleave(B, w)
            Lo, Xo, info_o = oracle.potrf_potrs_il(Af, Bf, n, nrhs, batch, w, layout, fill,
                                                   nthreads=NT)
            tA, tB = _dev(Af), _dev(Bf)
            info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
            bs.bs_potrf_potrs_batched_ex(tA, tB, info, layout, fill, interleave=w,
                                         shape=(batch, n, nrhs))
            Ag, Bg, infg = _host(tA), _host(tB), _host(info)
            assert np.array_equal(infg, info_o) and infg[batch // 2] == n, (n, w)
            ok = infg == 0
            for got, ref, shape in ((Ag, Lo, A.shape[1:]), (Bg, Xo, B.shape[1:])):
                # the systems that factored, bit for bit (the untouched triangle too)
                g2 = deinterleave(got, batch, w, shape)
                assert np.array_equal(g2[ok], deinterleave(ref, batch, w, shape)[ok]), (n, w)
                # the slots past the batch are never written
                pads = np.isnan(interleave(np.zeros((batch,) + shape), w))
                assert np.all(np.isnan(got[pads]))
            assert np.all(deinterleave(Bg, batch, w, B.shape[1:])[~ok] == 0)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_interleaved_with_contract_options(dtype, layout):
    """Interleaved layouts with a pivot threshold or the RUDA contract (one system per
    CTA, the element stride in every access): LU with tau 0.5 and with RUDA status codes,
    Cholesky under RUDA (-2 and a failing minor), against the oracle bit for bit."""
    from gen.workloads import deinterleave, interleave
    rng = np.random.default_rng(1919 + layout)
    batch = 21
    for n in (3, 16, 33, 64):
        for w in (4, 32):
            nrhs = int(rng.integers(1, 9))
            Al = rng.standard_normal((batch, n, n)).astype(dtype)
            Al[1, 0, 0] = np.inf
            Al[2, :, n // 2] = 0
            A, B = to_storage(Al, layout), to_storage(
                rng.standard_normal((batch, n, nrhs)).astype(dtype), layout)
            Af, Bf = interleave(A, w), interleave(B, w)
            for tau, ruda in ((0.5, 0), (1.0, 1)):
                So, Xo, ipo, info_o, tie = oracle.getrf_getrs_il(Af, Bf, n, nrhs, batch, w, layout,
                                                                 nthreads=NT, tau=tau, ruda=ruda)
                tA, tB = _dev(Af), _dev(Bf)
                ipiv = torch.full((Af.size // n,), SENT, dtype=torch.int32, device="cuda")
                info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
                bs.bs_getrf_getrs_batched_ex(tA, tB, ipiv, info, layout, tau,
                                             bs.BS_CONTRACT_RUDA if ruda else 0, interleave=w,
                                             shape=(batch, n, nrhs))
                Ag, Bg, ipg, infg = _host(tA), _host(tB), _host(ipiv), _host(info)
                clean = tie < 0
                assert np.array_equal(infg[clean], info_o[clean]), (n, w, tau, ruda)
                for got, ref, shape in ((Ag, So, A.shape[1:]), (Bg, Xo, B.shape[1:]),
                                        (ipg, ipo, (n,))):
                    g2, r2 = (deinterleave(got, batch, w, shape),
                              deinterleave(ref, batch, w, shape))
                    assert np.array_equal(g2[clean], r2[clean], equal_nan=True), (n, w, tau)
            G = rng.standard_normal((batch, n, n))
            Sl = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dtype)
            Sl[3, n - 1, 0] += 1.0
            Sl[4, n // 2, n // 2] = -1.0
            for fill in (bs.BS_LOWER, bs.BS_UPPER):
                Sa = interleave(to_storage(Sl, layout), w)
                Lo, Xo, info_o = oracle.potrf_potrs_il(Sa, Bf, n, nrhs, batch, w, layout, fill,
                                                       nthreads=NT, ruda=1)
                tA, tB = _dev(Sa), _dev(Bf)
                info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
                bs.bs_potrf_potrs_batched_ex(tA, tB, info, layout, fill, bs.BS_CONTRACT_RUDA,
                                             interleave=w, shape=(batch, n, nrhs))
                assert np.array_equal(_host(info), info_o) and info_o[3] == -2
                assert np.array_equal(_host(tA), Lo, equal_nan=True), (n, w, fill)
                assert np.array_equal(_host(tB), Xo, equal_nan=True), (n, w, fill)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_ruda_scaling(dtype, layout):
    """RUDA's max-abs scaling with U's scale restored: every order class (register-size,
    n > 32, n = 128), magnitudes far from 1, a power-of-two maximum, a singular system, a
    NaN (left unscaled), with the threshold, the RUDA contract and interleaving, against
    the oracle bit for bit."""
    from gen.workloads import deinterleave, interleave
    rng = np.random.default_rng(2020 + layout)
    batch = 13
    big = 1e15 if dtype == np.float32 else 1e150
    for n in (1, 2, 7, 16, 31, 32, 33, 64, 128):
        nrhs = int(rng.integers(1, 9))
        Al = rng.uniform(-1, 1, (batch, n, n)).astype(dtype)
        Al[0] *= dtype(3.7)
        Al[1] *= dtype(1.0 / big)
        Al[2] *= dtype(big)
        Al[3, 0, n - 1] = 4.0
        Al[4, :, n // 2] = 0
        Al[5, n - 1, 0] = np.nan
        A = to_storage(Al, layout)
        B = to_storage(rng.standard_normal((batch, n, nrhs)).astype(dtype), layout)
        for tau, ruda, w in ((1.0, 0, 0), (0.5, 0, 0), (1.0, 1, 0), (1.0, 0, 4)):
            if w:
                So, Xo, ipo, info_o, tie = oracle.getrf_getrs_il(
                    interleave(A, w), interleave(B, w), n, nrhs, batch, w, layout, nthreads=NT,
                    tau=tau, ruda=ruda, scale=1)
                tA, tB = _dev(interleave(A, w)), _dev(interleave(B, w))
                ipiv = torch.full((interleave(A, w).size // n,), SENT, dtype=torch.int32,
                                  device="cuda")
            else:
                So, Xo, ipo, info_o, tie = oracle.getrf_getrs_ex(A, B, layout, tau=tau,
                                                                 ruda=ruda, nthreads=NT,
                                                                 scale=1)
                tA, tB = _dev(A), _dev(B)
                ipiv = torch.full((batch, n), SENT, dtype=torch.int32, device="cuda")
            info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
            bs.bs_getrf_getrs_batched_ex(tA, tB, ipiv, info, layout, tau,
                                         bs.BS_CONTRACT_RUDA if ruda else 0, interleave=w,
                                         shape=(batch, n, nrhs), scaling=1)
            Ag, Bg, ipg, infg = _host(tA), _host(tB), _host(ipiv), _host(info)
            if w:
                So, Xo, ipo = (deinterleave(So, batch, w, A.shape[1:]),
                               deinterleave(Xo, batch, w, B.shape[1:]),
                               deinterleave(ipo, batch, w, (n,)))
                Ag, Bg, ipg = (deinterleave(Ag, batch, w, A.shape[1:]),
                               deinterleave(Bg, batch, w, B.shape[1:]),
                               deinterleave(ipg, batch, w, (n,)))
            clean = tie < 0
            assert clean.sum() >= batch - 4, (n, tau, ruda, w)
            assert np.array_equal(infg[clean], info_o[clean]), (n, tau, ruda, w)
            assert np.array_equal(ipg[clean], ipo[clean]), (n, tau, ruda, w)
            assert np.array_equal(Ag[clean], So[clean], equal_nan=True), (n, tau, ruda, w)
            assert np.array_equal(Bg[clean], Xo[clean], equal_nan=True), (n, tau, ruda, w)
