"""The documented limits, reached: 65,536 right-hand sides (the factor, then the solve
eight columns at a time) for the register LU, the one-CTA LU, the row-major reading, the
register and one-CTA Cholesky and the cluster Cholesky; against the CPU oracle bit for
bit; one more right-hand side is refused."""
import os

import numpy as np
import pytest
import torch

import dense_linear_solvers_gb300 as bs
import oracle
from gen.workloads import COL_MAJOR, ROW_MAJOR, to_storage

pytestmark = pytest.mark.gpu
NT = os.cpu_count() or 1
MAX_NRHS = 65536


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bs.lib()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


@pytest.mark.parametrize("dtype,n,layout", [(np.float32, 16, ROW_MAJOR),
                                            (np.float32, 16, COL_MAJOR),
                                            (np.float64, 100, ROW_MAJOR)])
def test_lu_max_right_hand_sides(dtype, n, layout):
    rng = np.random.default_rng(4141 + n + layout)
    batch = 2
    A = to_storage(rng.standard_normal((batch, n, n)).astype(dtype), layout)
    B = to_storage(rng.standard_normal((batch, n, MAX_NRHS)).astype(dtype), layout)
    Fo, Xo, ipo, info_o, tie = oracle.getrf_getrs(A, B, layout, nthreads=NT)
    assert np.all(tie < 0) and np.all(info_o == 0)
    tA, tB = _dev(A), _dev(B)
    ipiv = torch.zeros((batch, n), dtype=torch.int32, device="cuda")
    info = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    bs.bs_getrf_getrs_batched(tA, tB, ipiv, info, layout)
    torch.cuda.synchronize()
    assert np.array_equal(info.cpu().numpy(), info_o)
    assert np.array_equal(ipiv.cpu().numpy(), ipo)
    assert np.array_equal(tA.cpu().numpy(), Fo)
    assert np.array_equal(tB.cpu().numpy(), Xo)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_row_major_reading_max_right_hand_sides(dtype):
    rng = np.random.default_rng(4242)
    n, batch = 16, 2
    A = rng.standard_normal((batch, n, n)).astype(dtype)
    B = rng.standard_normal((batch, n, MAX_NRHS)).astype(dtype)
    So, Xo, ipo, info_o, tie = oracle.getrf_getrs_mirror(A, B, ROW_MAJOR, nthreads=NT)
    assert np.all(tie < 0)
    tA, tB = _dev(A), _dev(B)
    ipiv = torch.zeros((batch, n), dtype=torch.int32, device="cuda")
    info = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    bs.bs_getrf_getrs_batched_ex(tA, tB, ipiv, info, ROW_MAJOR, transposed_factor=1)
    torch.cuda.synchronize()
    assert np.array_equal(info.cpu().numpy(), info_o)
    assert np.array_equal(tA.cpu().numpy(), So)
    assert np.array_equal(tB.cpu().numpy(), Xo)


@pytest.mark.parametrize("n", [32, 100, 160])
def test_cholesky_max_right_hand_sides(n):
    rng = np.random.default_rng(4343 + n)
    batch = 2
    G = rng.standard_normal((batch, n, n))
    A = to_storage(G @ np.swapaxes(G, 1, 2) + n * np.eye(n), COL_MAJOR)
    B = to_storage(rng.standard_normal((batch, n, MAX_NRHS)), COL_MAJOR)
    Lo, Xo, info_o = oracle.potrf_potrs(A, B, COL_MAJOR, nthreads=NT)
    assert np.all(info_o == 0)
    tA, tB = _dev(A), _dev(B)
    info = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    bs.bs_potrf_potrs_batched(tA, tB, info, COL_MAJOR, bs.BS_LOWER)
    torch.cuda.synchronize()
    assert np.array_equal(info.cpu().numpy(), info_o)
    assert np.array_equal(tA.cpu().numpy(), Lo)
    assert np.array_equal(tB.cpu().numpy(), Xo)


def test_one_more_right_hand_side_is_refused():
    L = bs.lib()
    assert L.bs_getrf_getrs_supported(bs.BS_FP32, bs.BS_ROW_MAJOR, 16, MAX_NRHS) == 1
    assert L.bs_getrf_getrs_supported(bs.BS_FP32, bs.BS_ROW_MAJOR, 16, MAX_NRHS + 1) == 0
    assert L.bs_potrf_potrs_supported(bs.BS_FP64, bs.BS_COL_MAJOR, bs.BS_LOWER, 256,
                                      MAX_NRHS) == 1
    assert L.bs_potrf_potrs_supported(bs.BS_FP64, bs.BS_COL_MAJOR, bs.BS_LOWER, 256,
                                      MAX_NRHS + 1) == 0
