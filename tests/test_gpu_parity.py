"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Covers the five workloads at full size in the launch configuration the benchmark uses,
small batches spanning many blocks with a ragged tail, every supported order, both
layouts and dtypes, and the degenerate cases (singular pivots, planted indefinite
minors, NaN entries, empty batches). Criteria: tests/parity.py.
"""
import os

import numpy as np
import pytest
import torch

import dense_linear_solvers_gb300 as bs
import oracle
from gen import workloads as W
from gen.workloads import COL_MAJOR, ROW_MAJOR, to_storage
from tests import parity

pytestmark = pytest.mark.gpu
NT = os.cpu_count() or 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bs.lib()


def _log(name, rep):
    print(f"\n[{name}] " + " ".join(f"{k}={v}" for k, v in rep.items()))


# ------------------------------------------------------------------ the five workloads
@pytest.mark.parametrize("name,batch", [
    ("lu_f64_n8", None), ("lu_f32_n16", None), ("lu_f64_n64", None),
    ("lu_f64_n8", 37), ("lu_f32_n16", 1037), ("lu_f64_n64", 301),
])
def test_lu_workload(name, batch):
    d = W.make(name, batch)
    w = d["workload"]
    gpu = parity.gpu_lu(d["A"], d["B"], w.layout)
    orc = oracle.getrf_getrs(d["A"], d["B"], w.layout, nthreads=NT)
    rep = parity.check_lu(d["A"], d["B"], w.layout, gpu, orc, kappa=d.get("kappa"))
    for s, k in d["planted_info"].items():
        assert gpu[3][s] == k
    _log(f"{name} batch={d['batch']}", rep)


@pytest.mark.parametrize("batch", [None, 1000])
def test_chol_workload(batch):
    d = W.make("chol_f64_n32", batch)
    gpu = parity.gpu_chol(d["A"], d["B"], COL_MAJOR)
    orc = oracle.potrf_potrs(d["A"], d["B"], COL_MAJOR, nthreads=NT)
    rep = parity.check_chol(d["A"], d["B"], COL_MAJOR, gpu, orc)
    for s, k in d["planted_info"].items():
        assert gpu[2][s] == k
    assert rep["failed_systems"] == len(d["planted_info"])
    _log(f"chol_f64_n32 batch={d['batch']}", rep)


@pytest.mark.parametrize("batch", [None, 129])
def test_bdsv_workload(batch):
    d = W.make("bdsv_f64_32x8", batch)
    gpu = parity.gpu_bdsv(d["strips"], d["x"])
    orc = oracle.bdsv(d["strips"], d["x"], nthreads=NT)
    rep = parity.check_bdsv(d["strips"], d["x"], gpu, orc)
    _log(f"bdsv_f64_32x8 batch={d['batch']}", rep)


# ------------------------------------------------------------------ shape sweeps
@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_lu_every_order(dtype, layout):
    rng = np.random.default_rng(101 + layout)
    for n in range(1, 65):
        nrhs = int(rng.integers(1, 9))
        batch = 37
        A = to_storage(rng.standard_normal((batch, n, n)).astype(dtype), layout)
        B = to_storage(rng.standard_normal((batch, n, nrhs)).astype(dtype), layout)
        gpu = parity.gpu_lu(A, B, layout)
        orc = oracle.getrf_getrs(A, B, layout)
        parity.check_lu(A, B, layout, gpu, orc)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("layout", [ROW_MAJOR, COL_MAJOR])
def test_chol_every_order(dtype, layout):
    rng = np.random.default_rng(202 + layout)
    for n in range(1, 65):
        nrhs = int(rng.integers(1, 9))
        batch = 19
        G = rng.standard_normal((batch, n, n))
        Al = G @ np.swapaxes(G, 1, 2) + n * np.eye(n)
        if n > 2:
            Al[3, n // 2, n // 2] = -1.0       # one planted indefinite minor
        A = to_storage(Al.astype(dtype), layout)
        B = to_storage(rng.standard_normal((batch, n, nrhs)).astype(dtype), layout)
        gpu = parity.gpu_chol(A, B, layout)
        orc = oracle.potrf_potrs(A, B, layout)
        parity.check_chol(A, B, layout, gpu, orc)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_bdsv_every_block_size(dtype):
    rng = np.random.default_rng(303)
    for bsz in range(1, 9):
        for nbr in (1, 2, 3, 7):
            batch = 45
            strips = np.zeros((batch, nbr, bsz, 3 * bsz))
            C = rng.uniform(-0.5, 0.5, (batch, max(nbr - 1, 0), bsz, bsz)) / bsz
            M = rng.standard_normal((batch, nbr, bsz, bsz)) / np.sqrt(bsz)
            strips[:, :, :, bsz:2 * bsz] = M @ np.swapaxes(M, 2, 3) + 4.0 * np.eye(bsz)
            if nbr > 1:
                strips[:, :nbr - 1, :, 2 * bsz:] = C
                strips[:, 1:, :, :bsz] = np.swapaxes(C, 2, 3)
            xpad = np.zeros((batch, (nbr + 2) * bsz))
            xpad[:, bsz:(nbr + 1) * bsz] = rng.standard_normal((batch, nbr * bsz))
            xpad[:, :bsz] = 123.0       # pads must stay as they are
            xpad[:, (nbr + 1) * bsz:] = -5.0
            strips[:, :, :, 2 * bsz:] += 7.0 if nbr == 1 else 0.0  # RIGHT is never read
            strips[5, nbr - 1, bsz - 1, 2 * bsz - 1] = -50.0        # an indefinite last knot
            strips, xpad = strips.astype(dtype), xpad.astype(dtype)
            gpu = parity.gpu_bdsv(strips, xpad)
            orc = oracle.bdsv(strips, xpad)
            parity.check_bdsv(strips, xpad, gpu, orc)
            assert gpu[2][5] > 0


# ------------------------------------------------------------------ degenerate cases
@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_lu_singular_and_nan(dtype):
    rng = np.random.default_rng(404)
    for n in (3, 8, 16, 32, 40, 64):
        batch = 3 * n + 5
        A = rng.uniform(-1, 1, (batch, n, n)).astype(dtype)
        for j in range(n):
            A[j, :, j] = 0                      # a zero column at every position
        A[n, :, :] = 0                          # all zero: info = 1
        A[n + 1, 1] = A[n + 1, 0]               # two equal rows
        A[n + 2, n // 2, n // 3] = np.nan       # a NaN entry
        A[n + 3, 0, 0] = np.nan                 # a NaN in the first pivot position
        A[n + 4, :, 0] = np.finfo(dtype).smallest_subnormal  # subnormal pivot column
        B = rng.uniform(-1, 1, (batch, n, 2)).astype(dtype)
        gpu = parity.gpu_lu(A, B, ROW_MAJOR)
        orc = oracle.getrf_getrs(A, B, ROW_MAJOR)
        nan = np.zeros(batch, bool)
        nan[[n + 2, n + 3]] = True
        fin = ~nan
        parity.check_lu(A[fin], B[fin], ROW_MAJOR, tuple(g[fin] for g in gpu),
                        tuple(o[fin] for o in orc))
        for j in range(n):
            assert gpu[3][j] == j + 1
        assert gpu[3][n] == 1 and gpu[3][n + 4] == 1
        # NaN inputs: the same decisions and the same (possibly NaN) numbers as the oracle
        assert np.array_equal(gpu[3][nan], orc[3][nan])
        assert np.array_equal(gpu[2][nan], orc[2][nan])
        assert np.array_equal(gpu[1][nan], orc[1][nan], equal_nan=True)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_lu_layout_invariance(dtype):
    """Row- and column-major storage of the same matrices: the same pivots, info and,
    the arithmetic being the same, bitwise equal factors and solutions."""
    rng = np.random.default_rng(505)
    for n in (5, 16, 32, 48, 64):
        Al = rng.standard_normal((50, n, n)).astype(dtype)
        Bl = rng.standard_normal((50, n, 3)).astype(dtype)
        r = parity.gpu_lu(to_storage(Al, ROW_MAJOR), to_storage(Bl, ROW_MAJOR), ROW_MAJOR)
        c = parity.gpu_lu(to_storage(Al, COL_MAJOR), to_storage(Bl, COL_MAJOR), COL_MAJOR)
        assert np.array_equal(r[2], c[2]) and np.array_equal(r[3], c[3])
        assert np.array_equal(r[0], np.swapaxes(c[0], 1, 2))
        assert np.array_equal(r[1], np.swapaxes(c[1], 1, 2))


def test_empty_batch_launches_nothing():
    dev = torch.device("cuda")
    A = torch.zeros((0, 16, 16), device=dev)
    B = torch.zeros((0, 16, 4), device=dev)
    bs.bs_getrf_getrs_batched(A, B, torch.zeros((0, 16), dtype=torch.int32, device=dev),
                              torch.zeros(0, dtype=torch.int32, device=dev))
    Bc = torch.zeros((0, 4, 16), dtype=torch.float64, device=dev)  # column-major storage
    bs.bs_potrf_potrs_batched(A.double(), Bc, torch.zeros(0, dtype=torch.int32, device=dev),
                              COL_MAJOR)
    S = torch.zeros((0, 32, 8, 24), dtype=torch.float64, device=dev)
    X = torch.zeros((0, 34 * 8), dtype=torch.float64, device=dev)
    bs.bs_bdsv_batched(S, X, torch.zeros(0, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()


def test_unsupported_shape_is_an_error():
    dev = torch.device("cuda")
    A = torch.zeros((2, 129, 129), device=dev)
    B = torch.zeros((2, 129, 1), device=dev)
    with pytest.raises(bs.BsolveError) as e:
        bs.bs_getrf_getrs_batched(A, B, torch.zeros((2, 129), dtype=torch.int32, device=dev),
                                  torch.zeros(2, dtype=torch.int32, device=dev))
    assert e.value.status == bs.BS_ERR_UNSUPPORTED
