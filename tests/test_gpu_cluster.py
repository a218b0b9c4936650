"""Cholesky for 128 < n <= 256 (the factor on a cluster of four CTAs, the triangle's tiles
spread over their shared memory; the solve one CTA per system) against the CPU oracle:
factor and X bit for bit where the factorization succeeds, info exact on planted
indefinite minors (in the first tile, deep inside, in the last partial tile), X zero on
failure, the other triangle never read (NaN there) nor written, both storage orders,
both fills, ragged orders and right-hand-side counts, the split calls."""
import numpy as np
import pytest
import torch

import dense_linear_solvers_gb300 as bs
import oracle
from gen.workloads import COL_MAJOR, ROW_MAJOR, from_storage, to_storage
from tests import parity

pytestmark = pytest.mark.gpu
SENT = -7


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bs.lib()


def _spd(rng, batch, n, dtype, plant):
    G = rng.standard_normal((batch, n, n))
    Al = G @ np.swapaxes(G, 1, 2) + n * np.eye(n)
    for s, k in plant.items():
        Al[s, k, k] = -1.0
    return Al.astype(dtype)


def _with_nan_outside(Al, fill):
    """The logical matrix with the triangle the call must not read set to NaN."""
    A = Al.copy()
    n = A.shape[1]
    iu = np.triu_indices(n, 1) if fill == bs.BS_LOWER else np.tril_indices(n, -1)
    A[:, iu[0], iu[1]] = np.nan
    return A


def _run(A, B, layout, fill):
    tA = torch.from_numpy(np.ascontiguousarray(A)).cuda()
    tB = torch.from_numpy(np.ascontiguousarray(B)).cuda()
    info = torch.full((A.shape[0],), SENT, dtype=torch.int32, device="cuda")
    bs.bs_potrf_potrs_batched(tA, tB, info, layout, fill)
    torch.cuda.synchronize()
    return tA.cpu().numpy(), tB.cpu().numpy(), info.cpu().numpy()


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
@pytest.mark.parametrize("fill", [bs.BS_LOWER, bs.BS_UPPER])
def test_cluster_cholesky_matches_oracle(dtype, layout, fill):
    rng = np.random.default_rng(909 + 2 * layout + fill)
    for n in (129, 150, 160, 192, 223, 256):
        nrhs = int(rng.integers(1, 12))
        batch = 7
        plant = {1: 3, 3: n - 1, 5: min(n - 1, 140)}
        Al = _spd(rng, batch, n, dtype, plant)
        A = to_storage(_with_nan_outside(Al, fill), layout)
        B = to_storage(rng.standard_normal((batch, n, nrhs)).astype(dtype), layout)
        Fg, Xg, infg = _run(A, B, layout, fill)
        Fo, Xo, info_o = oracle.potrf_potrs(A, B, layout, fill=fill)
        assert np.array_equal(infg, info_o), (n, infg, info_o)
        for s, k in plant.items():
            assert infg[s] == k + 1
        ok = info_o == 0
        # the whole factor array, the unread triangle (NaN) included, and X: bit for bit
        assert np.array_equal(Fg[ok], Fo[ok], equal_nan=True), n
        assert np.array_equal(Xg[ok], Xo[ok]), n
        assert np.all(Xg[~ok] == 0)
        # the unread triangle is untouched on failed systems too
        Fl = from_storage(Fg, layout)
        iu = np.triu_indices(n, 1) if fill == bs.BS_LOWER else np.tril_indices(n, -1)
        assert np.all(np.isnan(Fl[:, iu[0], iu[1]]))


def test_cluster_cholesky_backward_error():
    """A larger batch of one order with the stated criteria (tests/parity.py)."""
    rng = np.random.default_rng(910)
    n, batch = 200, 64
    Al = _spd(rng, batch, n, np.float64, {7: 50})
    A = to_storage(Al, COL_MAJOR)
    B = to_storage(rng.standard_normal((batch, n, 2)), COL_MAJOR)
    gpu = parity.gpu_chol(A, B, COL_MAJOR)
    orc = oracle.potrf_potrs(A, B, COL_MAJOR)
    rep = parity.check_chol(A, B, COL_MAJOR, gpu, orc)
    assert rep["failed_systems"] == 1


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_cluster_split_calls(dtype, layout):
    """potrf alone = the fused call's factor; potrs from the oracle's factor = the
    oracle's X; potrf then potrs = the fused call."""
    rng = np.random.default_rng(911 + layout)
    n, batch, nrhs = 176, 5, 9
    Al = _spd(rng, batch, n, dtype, {2: 33})
    A = to_storage(Al, layout)
    B = to_storage(rng.standard_normal((batch, n, nrhs)).astype(dtype), layout)
    tA = torch.from_numpy(np.ascontiguousarray(A)).cuda()
    info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
    bs.bs_potrf_batched(tA, info, layout)
    Lo, info_o = oracle.potrf(A, layout)
    Lg = tA.cpu().numpy()
    assert np.array_equal(info.cpu().numpy(), info_o)
    ok = info_o == 0
    assert np.array_equal(Lg[ok], Lo[ok])
    tB = torch.from_numpy(np.ascontiguousarray(B)).cuda()
    bs.bs_potrs_batched(torch.from_numpy(Lo).cuda(), tB, layout)
    Xo = oracle.potrs(Lo, B, layout)
    assert np.array_equal(tB.cpu().numpy()[ok], Xo[ok])
    Ff, Xf, inff = _run(A, B, layout, bs.BS_LOWER)
    assert np.array_equal(Ff[ok], Lg[ok]) and np.array_equal(inff, info.cpu().numpy())
    tB2 = torch.from_numpy(np.ascontiguousarray(B)).cuda()
    bs.bs_potrs_batched(torch.from_numpy(Lg).cuda(), tB2, layout)
    assert np.array_equal(tB2.cpu().numpy()[ok], Xf[ok])


def test_cluster_orders_refused_where_unsupported():
    """Beyond one CTA, the contract options and interleaved layouts are refused; LU
    stays at n <= 128."""
    L = bs.lib()
    assert L.bs_potrf_potrs_supported(bs.BS_FP64, 1, 0, 256, 1) == 1
    assert L.bs_potrf_potrs_supported(bs.BS_FP64, 1, 0, 257, 1) == 0
    assert L.bs_getrf_getrs_supported(bs.BS_FP64, 1, 129, 1) == 0
    A = torch.zeros((4, 160, 160), dtype=torch.float64, device="cuda")
    B = torch.zeros((4, 1, 160), dtype=torch.float64, device="cuda")   # column-major
    info = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError):
        bs.bs_potrf_potrs_batched_ex(A, B, info, COL_MAJOR, bs.BS_LOWER,
                                     status_contract=bs.BS_CONTRACT_RUDA)
