"""Factor once, solve per right-hand side, and the block-tridiagonal matvec: the CUDA path
(through the C ABI) against the CPU oracle, element by element.

  * getrf / potrf / bdsv_factor leave the oracle's factor, pivots and info bit for bit
    (LU: on every step before the oracle's first near tie);
  * getrs / potrs / bdsv_solve, given the oracle's factor, leave the oracle's X bit for
    bit; given the GPU's own factor they reproduce the GPU's fused call bit for bit;
  * bdmv equals the oracle's matvec bit for bit and leaves the pad blocks of y alone.
Shapes: the benchmark workloads at full size, every supported order and block size with
both layouts and dtypes, ragged batches, singular and indefinite systems, pivot entries
out of range.
"""
import os

import numpy as np
import pytest
import torch

import dense_linear_solvers_gb300 as bs
import oracle
from gen import workloads as W
from gen.workloads import COL_MAJOR, ROW_MAJOR, from_storage, to_storage
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


# ------------------------------------------------------------------ LU
def gpu_getrf(A, layout):
    tA = _dev(A)
    batch, n = A.shape[0], A.shape[1]
    ipiv = torch.full((batch, n), SENT, dtype=torch.int32, device="cuda")
    info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
    bs.bs_getrf_batched(tA, ipiv, info, layout)
    return _host(tA), _host(ipiv), _host(info)


def gpu_getrs(LU, ipiv, B, layout):
    tB = _dev(B)
    bs.bs_getrs_batched(_dev(LU), _dev(ipiv.astype(np.int32)), tB, layout)
    return _host(tB)


def check_getrf(A, layout, gpu, orc):
    LUg, ipg, infg = gpu
    LUo, ipo, info_o, tie = orc
    n = A.shape[1]
    assert np.all(ipg != SENT) and np.all(infg != SENT)
    clean = tie < 0
    info_cmp = clean | ((info_o > 0) & (info_o - 1 < tie))
    assert np.array_equal(infg[info_cmp], info_o[info_cmp])
    steps = np.where(clean, n, tie)
    mask = np.arange(n)[None, :] < steps[:, None]
    assert not np.any(mask & (ipg != ipo))
    assert np.array_equal(LUg[clean], LUo[clean])
    return clean


def _lu_case(A, B, layout):
    """getrf and getrs against the oracle, and the GPU's own factor + solve against the
    GPU's fused call."""
    orc_f = oracle.getrf(A, layout, nthreads=NT)
    gpu_f = gpu_getrf(A, layout)
    clean = check_getrf(A, layout, gpu_f, orc_f)
    # the solve alone, from the oracle's factor: the oracle's X bit for bit
    Xo = oracle.getrs(orc_f[0], orc_f[1], B, layout, nthreads=NT)
    Xg = gpu_getrs(orc_f[0], orc_f[1], B, layout)
    ok = orc_f[2] == 0
    assert np.array_equal(Xg[ok], Xo[ok])
    # factor + solve on the GPU = the fused GPU call
    LUf, Xf, ipf, inff = parity.gpu_lu(A, B, layout)
    Xs = gpu_getrs(gpu_f[0], gpu_f[1], B, layout)
    assert np.array_equal(gpu_f[0], LUf) and np.array_equal(gpu_f[1], ipf)
    assert np.array_equal(gpu_f[2], inff)
    good = inff == 0
    assert np.array_equal(Xs[good], Xf[good])
    return int(clean.sum())


@pytest.mark.parametrize("name,batch", [("lu_f32_n16", None), ("lu_f64_n8", None),
                                        ("lu_f64_n64", None), ("lu_f64_n64", 301),
                                        ("lu_f32_n16", 1037)])
def test_getrf_getrs_workload(name, batch):
    d = W.make(name, batch)
    _lu_case(d["A"], d["B"], d["workload"].layout)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_getrf_getrs_every_order(dtype, layout):
    rng = np.random.default_rng(505 + layout)
    for n in range(1, 65):
        nrhs = int(rng.integers(1, 9))
        Al = rng.standard_normal((37, n, n)).astype(dtype)
        if n > 1:
            Al[5, :, n // 2] = 0          # singular: info > 0
        A = to_storage(Al, layout)
        B = to_storage(rng.standard_normal((37, n, nrhs)).astype(dtype), layout)
        _lu_case(A, B, layout)


def test_getrs_reuses_one_factor():
    """One factor, several right-hand-side sets: each solve equals its fused call."""
    rng = np.random.default_rng(506)
    A = rng.standard_normal((300, 16, 16)).astype(np.float32)
    LU, ipiv, info = gpu_getrf(A, ROW_MAJOR)
    for rep in range(3):
        B = rng.standard_normal((300, 16, 4)).astype(np.float32)
        _, Xf, _, _ = parity.gpu_lu(A, B, ROW_MAJOR)
        assert np.array_equal(gpu_getrs(LU, ipiv, B, ROW_MAJOR), Xf)


def test_getrs_pivot_entry_out_of_range_swaps_nothing():
    rng = np.random.default_rng(507)
    for n in (5, 16, 40):
        LU = rng.standard_normal((9, n, n)) + 4 * np.eye(n)
        ipiv = np.stack([rng.integers(k, n, size=9) for k in range(n)], axis=1).astype(np.int32) + 1
        ipiv[1, 0] = 0
        ipiv[2, n - 1] = n + 5
        ipiv[3, :] = -3
        clean = ipiv.copy()
        bad = (clean < 1) | (clean > n)
        clean[bad] = (np.arange(n)[None, :].repeat(9, 0) + 1)[bad]
        B = rng.standard_normal((9, n, 2))
        Xo = oracle.getrs(LU, clean, B, ROW_MAJOR)
        assert np.array_equal(gpu_getrs(LU, ipiv, B, ROW_MAJOR), Xo)


# ------------------------------------------------------------------ Cholesky
def gpu_potrf(A, layout):
    tA = _dev(A)
    info = torch.full((A.shape[0],), SENT, dtype=torch.int32, device="cuda")
    bs.bs_potrf_batched(tA, info, layout)
    return _host(tA), _host(info)


def gpu_potrs(L, B, layout):
    tB = _dev(B)
    bs.bs_potrs_batched(_dev(L), tB, layout)
    return _host(tB)


def _chol_case(A, B, layout):
    Lo, info_o = oracle.potrf(A, layout, nthreads=NT)
    Lg, infg = gpu_potrf(A, layout)
    assert np.array_equal(infg, info_o)
    ok = info_o == 0
    assert np.array_equal(Lg[ok], Lo[ok], equal_nan=True)   # the strict upper triangle too
    Xo = oracle.potrs(Lo, B, layout, nthreads=NT)
    Xg = gpu_potrs(Lo, B, layout)
    assert np.array_equal(Xg[ok], Xo[ok])
    Lf, Xf, inff = parity.gpu_chol(A, B, layout)
    assert np.array_equal(Lg[ok], Lf[ok], equal_nan=True) and np.array_equal(infg, inff)
    assert np.array_equal(gpu_potrs(Lg, B, layout)[ok], Xf[ok])


@pytest.mark.parametrize("batch", [None, 1000])
def test_potrf_potrs_workload(batch):
    d = W.make("chol_f64_n32", batch)
    _chol_case(d["A"], d["B"], COL_MAJOR)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_potrf_potrs_every_order(dtype, layout):
    rng = np.random.default_rng(606 + layout)
    for n in range(1, 65):
        nrhs = int(rng.integers(1, 9))
        G = rng.standard_normal((19, n, n))
        Al = G @ np.swapaxes(G, 1, 2) + n * np.eye(n)
        if n > 2:
            Al[3, n // 2, n // 2] = -1.0
        Al[7][np.triu_indices(n, 1)] = np.nan    # the upper triangle is never read
        A = to_storage(Al.astype(dtype), layout)
        B = to_storage(rng.standard_normal((19, n, nrhs)).astype(dtype), layout)
        _chol_case(A, B, layout)


@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
@pytest.mark.parametrize("fill", [bs.BS_LOWER, bs.BS_UPPER])
def test_potrs_fp64_one_rhs_every_order(layout, fill):
    """FP64 potrs with one right-hand side runs one system per lane: every order 1..32,
    both storage orders and fills, a batch of several warps and blocks with a ragged
    tail, the unread triangle NaN; X equals the oracle's bit for bit."""
    rng = np.random.default_rng(1818 + 2 * layout + fill)
    batch = 197
    for n in range(1, 33):
        G = rng.standard_normal((batch, n, n))
        Al = G @ np.swapaxes(G, 1, 2) + n * np.eye(n)
        A = to_storage(Al, layout)
        Lo, info_o = oracle.potrf(A, layout, fill=fill, nthreads=NT)
        assert np.all(info_o == 0)
        tri = np.triu_indices(n, 1) if fill == bs.BS_LOWER else np.tril_indices(n, -1)
        Ll = from_storage(Lo, layout).copy()
        Ll[:, tri[0], tri[1]] = np.nan
        Ln = to_storage(Ll, layout)
        B = to_storage(rng.standard_normal((batch, n, 1)), layout)
        Xo = oracle.potrs(Ln, B, layout, fill=fill, nthreads=NT)
        tB = _dev(B)
        bs.bs_potrs_batched(_dev(Ln), tB, layout, fill)
        assert np.array_equal(_host(tB), Xo), n


# ------------------------------------------------------------------ bdsv
def gpu_bdsv_factor(strips):
    tS = _dev(strips)
    info = torch.full((strips.shape[0],), SENT, dtype=torch.int32, device="cuda")
    bs.bs_bdsv_factor_batched(tS, info)
    return _host(tS), _host(info)


def gpu_bdsv_solve(strips, xpad):
    tX = _dev(xpad)
    bs.bs_bdsv_solve_batched(_dev(strips), tX)
    return _host(tX)


def _bdsv_case(strips, xpad):
    So, info_o = oracle.bdsv_factor(strips, nthreads=NT)
    Sg, infg = gpu_bdsv_factor(strips)
    assert np.array_equal(infg, info_o)
    ok = info_o == 0
    assert np.array_equal(Sg[ok], So[ok])
    Xo = oracle.bdsv_solve(So, xpad, nthreads=NT)
    Xg = gpu_bdsv_solve(So, xpad)
    assert np.array_equal(Xg[ok], Xo[ok])
    Sf, Xf, inff = parity.gpu_bdsv(strips, xpad)
    assert np.array_equal(infg, inff) and np.array_equal(Sg[ok], Sf[ok])
    assert np.array_equal(gpu_bdsv_solve(Sg, xpad)[ok], Xf[ok])


@pytest.mark.parametrize("batch", [None, 129])
def test_bdsv_split_workload(batch):
    d = W.make("bdsv_f64_32x8", batch)
    _bdsv_case(d["strips"], d["x"])


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_bdsv_split_every_block_size(dtype):
    rng = np.random.default_rng(707)
    for bsz in range(1, 9):
        for nbr in (1, 2, 3, 7):
            strips = np.zeros((45, nbr, bsz, 3 * bsz))
            M = rng.standard_normal((45, nbr, bsz, bsz)) / np.sqrt(bsz)
            strips[:, :, :, bsz:2 * bsz] = M @ np.swapaxes(M, 2, 3) + 3.0 * np.eye(bsz)
            if nbr > 1:
                C = rng.uniform(-0.5, 0.5, (45, nbr - 1, bsz, bsz)) / bsz
                strips[:, :nbr - 1, :, 2 * bsz:] = C
                strips[:, 1:, :, :bsz] = np.swapaxes(C, 2, 3)
            strips[6, nbr - 1, bsz - 1, 2 * bsz - 1] = -1.0     # a failing knot
            xpad = np.zeros((45, (nbr + 2) * bsz))
            xpad[:, bsz:(nbr + 1) * bsz] = rng.standard_normal((45, nbr * bsz))
            _bdsv_case(strips.astype(dtype), xpad.astype(dtype))


# ------------------------------------------------------------------ bdmv
def gpu_bdmv(strips, xpad, y0):
    tY = _dev(y0)
    bs.bs_bdmv_batched(_dev(strips), _dev(xpad), tY)
    return _host(tY)


def test_bdmv_workload_full_size():
    d = W.make("bdsv_f64_32x8")
    strips, xpad = d["strips"], d["x"]
    y0 = np.full_like(xpad, 3.5)
    yg = gpu_bdmv(strips, xpad, y0)
    yo = oracle.bdmv(strips, xpad, y0, nthreads=NT)
    assert np.array_equal(yg, yo)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_bdmv_every_block_size(dtype):
    rng = np.random.default_rng(808)
    for bsz in range(1, 9):
        for nbr in (1, 2, 5, 33):
            batch = 67
            strips = rng.standard_normal((batch, nbr, bsz, 3 * bsz)).astype(dtype)
            xpad = rng.standard_normal((batch, (nbr + 2) * bsz)).astype(dtype)
            xpad[:, :bsz] = 0
            xpad[:, (nbr + 1) * bsz:] = 0
            y0 = np.full_like(xpad, -2.25)
            yg = gpu_bdmv(strips, xpad, y0)
            yo = oracle.bdmv(strips, xpad, y0)
            assert np.array_equal(yg, yo), (bsz, nbr)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_bdmv_two_outputs(dtype):
    """The second matvec form stores the oracle's bdmv values into both outputs (the pad
    blocks of each keep what they held); at the full workload size and over every block
    size."""
    rng = np.random.default_rng(818)
    cases = [(W.make("bdsv_f64_32x8")["strips"], W.make("bdsv_f64_32x8")["x"])] \
        if dtype == np.float64 else []
    for bsz in (1, 3, 8):
        for nbr in (1, 5, 33):
            strips = rng.standard_normal((61, nbr, bsz, 3 * bsz)).astype(dtype)
            xpad = rng.standard_normal((61, (nbr + 2) * bsz)).astype(dtype)
            xpad[:, :bsz] = 0
            xpad[:, (nbr + 1) * bsz:] = 0
            cases.append((strips, xpad))
    for strips, xpad in cases:
        y1, y2 = np.full_like(xpad, 3.5), np.full_like(xpad, -1.25)
        t1, t2 = _dev(y1), _dev(y2)
        bs.bs_bdmv2_batched(_dev(strips), _dev(xpad), t1, t2)
        assert np.array_equal(_host(t1), oracle.bdmv(strips, xpad, y1, nthreads=NT))
        assert np.array_equal(_host(t2), oracle.bdmv(strips, xpad, y2, nthreads=NT))


# ------------------------------------------------------------------ Cholesky, upper fill
@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_cholesky_upper_fill_every_order(dtype, layout):
    """Upper fill (A = U^T U): the fused call, potrf and potrs leave the oracle's U, info
    and X bit for bit; the strict lower triangle (NaN here) is neither read nor written."""
    rng = np.random.default_rng(909 + layout)
    for n in range(1, 65):
        nrhs = int(rng.integers(1, 9))
        G = rng.standard_normal((23, n, n))
        Al = G @ np.swapaxes(G, 1, 2) + n * np.eye(n)
        if n > 2:
            Al[4, n // 2, n // 2] = -1.0
        il = np.tril_indices(n, -1)
        Al[:, il[0], il[1]] = np.nan
        A = to_storage(Al.astype(dtype), layout)
        B = to_storage(rng.standard_normal((23, n, nrhs)).astype(dtype), layout)
        Uo, Xo, info_o = oracle.potrf_potrs(A, B, layout, nthreads=NT, fill=oracle.UPPER)
        tA, tB = _dev(A), _dev(B)
        info = torch.full((23,), SENT, dtype=torch.int32, device="cuda")
        bs.bs_potrf_potrs_batched(tA, tB, info, layout, bs.BS_UPPER)
        Ug, Xg, infg = _host(tA), _host(tB), _host(info)
        assert np.array_equal(infg, info_o)
        ok = info_o == 0
        assert np.array_equal(Ug[ok], Uo[ok], equal_nan=True)
        assert np.array_equal(Xg, Xo)                    # failed systems: zeros on both
        # the halves
        tA2 = _dev(A)
        info2 = torch.full((23,), SENT, dtype=torch.int32, device="cuda")
        bs.bs_potrf_batched(tA2, info2, layout, bs.BS_UPPER)
        assert np.array_equal(_host(info2), info_o)
        assert np.array_equal(_host(tA2)[ok], Uo[ok], equal_nan=True)
        tB2 = _dev(B)
        bs.bs_potrs_batched(_dev(Uo), tB2, layout, bs.BS_UPPER)
        Xs = _host(tB2)
        Xso = oracle.potrs(Uo, B, layout, fill=oracle.UPPER)
        assert np.array_equal(Xs[ok], Xso[ok])
        assert np.array_equal(Xs[ok], Xo[ok])


# ------------------------------------------------------------------ more right-hand sides
@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_many_right_hand_sides(dtype, layout):
    """nrhs > 8: the fused calls run as factor + chunked solve and still leave the oracle's
    fused results bit for bit (X zero where info != 0); getrs/potrs take the right-hand
    sides eight at a time."""
    rng = np.random.default_rng(1010 + layout)
    for n, nrhs in ((1, 9), (5, 13), (16, 40), (31, 17), (33, 9), (64, 24)):
        Al = rng.standard_normal((29, n, n)).astype(dtype)
        if n > 1:
            Al[3, :, n - 1] = 0
        A = to_storage(Al, layout)
        B = to_storage(rng.standard_normal((29, n, nrhs)).astype(dtype), layout)
        LUo, Xo, ipo, info_o, tie = oracle.getrf_getrs(A, B, layout, nthreads=NT)
        LUg, Xg, ipg, infg = parity.gpu_lu(A, B, layout)
        clean = tie < 0
        assert np.array_equal(infg[clean], info_o[clean])
        assert np.array_equal(LUg[clean], LUo[clean]) and np.array_equal(Xg[clean], Xo[clean])
        assert np.all(Xg[infg != 0] == 0)
        Xs = gpu_getrs(LUo, ipo, B, layout)
        ok = info_o == 0
        assert np.array_equal(Xs[ok], oracle.getrs(LUo, ipo, B, layout)[ok])
        # Cholesky, both fills
        G = rng.standard_normal((29, n, n))
        S = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dtype)
        if n > 2:
            S[5, 1, 1] = -1.0
        As = to_storage(S, layout)
        for fill in (bs.BS_LOWER, bs.BS_UPPER):
            Lo, Xco, inf_co = oracle.potrf_potrs(As, B, layout, nthreads=NT, fill=fill)
            tA, tB = _dev(As), _dev(B)
            info = torch.full((29,), SENT, dtype=torch.int32, device="cuda")
            bs.bs_potrf_potrs_batched(tA, tB, info, layout, fill)
            okc = inf_co == 0
            assert np.array_equal(_host(info), inf_co)
            assert np.array_equal(_host(tA)[okc], Lo[okc])
            assert np.array_equal(_host(tB), Xco)
            tB2 = _dev(B)
            bs.bs_potrs_batched(_dev(Lo), tB2, layout, fill)
            assert np.array_equal(_host(tB2)[okc], Xco[okc])


@pytest.mark.parametrize("dtype,layout,n,nrhs", [(np.float32, ROW_MAJOR, 16, 1003),
                                                (np.float64, COL_MAJOR, 64, 257)])
def test_hundreds_of_right_hand_sides(dtype, layout, n, nrhs):
    """Hundreds of right-hand sides (a ragged last chunk of 8): the fused LU and Cholesky
    calls still leave the oracle's fused results bit for bit."""
    rng = np.random.default_rng(1212 + layout)
    Al = rng.standard_normal((5, n, n)).astype(dtype)
    Al[2, :, n // 2] = 0
    A = to_storage(Al, layout)
    B = to_storage(rng.standard_normal((5, n, nrhs)).astype(dtype), layout)
    LUo, Xo, ipo, info_o, tie = oracle.getrf_getrs(A, B, layout, nthreads=NT)
    LUg, Xg, ipg, infg = parity.gpu_lu(A, B, layout)
    clean = tie < 0
    assert np.array_equal(infg[clean], info_o[clean]) and info_o[2] == n // 2 + 1
    assert np.array_equal(LUg[clean], LUo[clean]) and np.array_equal(Xg[clean], Xo[clean])
    G = rng.standard_normal((5, n, n))
    As = to_storage((G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dtype), layout)
    Lo, Xco, inf_co = oracle.potrf_potrs(As, B, layout, nthreads=NT)
    tA, tB = _dev(As), _dev(B)
    info = torch.full((5,), SENT, dtype=torch.int32, device="cuda")
    bs.bs_potrf_potrs_batched(tA, tB, info, layout, bs.BS_LOWER)
    assert np.array_equal(_host(info), inf_co) and np.all(inf_co == 0)
    assert np.array_equal(_host(tA), Lo) and np.array_equal(_host(tB), Xco)


# ------------------------------------------------------------------ orders 65..128
@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_orders_up_to_128(dtype, layout):
    """One system per CTA up to n = 128: the fused calls, the factor calls and the solves
    against the oracle, LU with a singular system, Cholesky (both fills) with an indefinite
    one."""
    rng = np.random.default_rng(1111 + layout)
    for n, nrhs in ((65, 3), (80, 8), (97, 1), (127, 12), (128, 5)):
        batch = 9
        Al = rng.standard_normal((batch, n, n)).astype(dtype)
        Al[2, :, n // 3] = 0
        A = to_storage(Al, layout)
        B = to_storage(rng.standard_normal((batch, n, nrhs)).astype(dtype), layout)
        LUo, Xo, ipo, info_o, tie = oracle.getrf_getrs(A, B, layout, nthreads=NT)
        LUg, Xg, ipg, infg = parity.gpu_lu(A, B, layout)
        clean = tie < 0
        assert np.array_equal(infg[clean], info_o[clean])
        assert np.array_equal(LUg[clean], LUo[clean]) and np.array_equal(Xg[clean], Xo[clean])
        assert np.all(Xg[infg != 0] == 0)
        _lu_case(A, B, layout)
        G = rng.standard_normal((batch, n, n))
        S = (G @ np.swapaxes(G, 1, 2) + n * np.eye(n)).astype(dtype)
        S[4, n // 2, n // 2] = -1.0
        As = to_storage(S, layout)
        for fill in (bs.BS_LOWER, bs.BS_UPPER):
            Lo, Xco, inf_co = oracle.potrf_potrs(As, B, layout, nthreads=NT, fill=fill)
            tA, tB = _dev(As), _dev(B)
            info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
            bs.bs_potrf_potrs_batched(tA, tB, info, layout, fill)
            okc = inf_co == 0
            assert np.array_equal(_host(info), inf_co)
            assert np.array_equal(_host(tA)[okc], Lo[okc]) and np.array_equal(_host(tB), Xco)
            tB2 = _dev(B)
            bs.bs_potrs_batched(_dev(Lo), tB2, layout, fill)
            assert np.array_equal(_host(tB2)[okc], Xco[okc])
