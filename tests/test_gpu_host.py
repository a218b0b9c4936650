"""Host-resident batches (bs_*_batched_host): the fused calls on pinned host arrays,
copied in and out by chunks on two streams. Results must equal the device calls' bit for
bit (the same kernels on the same systems, only the chunking differs), for ragged last
chunks, one-system chunks and a chunk larger than the batch, and at the benchmark's full
size; each case is also checked against the CPU oracle.
"""
import os

import numpy as np
import pytest
import torch

import dense_linear_solvers_gb300 as bs
import oracle
from gen import workloads as W
from gen.workloads import COL_MAJOR
from tests import parity

pytestmark = pytest.mark.gpu
NT = os.cpu_count() or 1
SENT = parity.SENTINEL


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bs.lib()


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def host_lu(A, B, layout, chunk):
    tA, tB = _pinned(A), _pinned(B)
    ipiv = torch.full((A.shape[0], A.shape[1]), SENT, dtype=torch.int32).pin_memory()
    info = torch.full((A.shape[0],), SENT, dtype=torch.int32).pin_memory()
    bs.bs_getrf_getrs_batched_host(tA, tB, ipiv, info, layout, chunk=chunk)
    return tA.numpy(), tB.numpy(), ipiv.numpy(), info.numpy()


@pytest.mark.parametrize("name,batch,chunk", [
    ("lu_f32_n16", 1037, 100), ("lu_f32_n16", 37, 1), ("lu_f32_n16", 500, 4096),
    ("lu_f64_n8", None, 333), ("lu_f64_n64", 301, 64), ("lu_f32_n16", None, 8192),
])
def test_host_lu(name, batch, chunk):
    d = W.make(name, batch)
    w = d["workload"]
    dev = parity.gpu_lu(d["A"], d["B"], w.layout)
    got = host_lu(d["A"], d["B"], w.layout, chunk)
    for g, r in zip(got, dev):
        assert np.array_equal(g, r, equal_nan=True), (name, batch, chunk)
    if d["A"].shape[0] <= 2048:
        orc = oracle.getrf_getrs(d["A"], d["B"], w.layout, nthreads=NT)
        parity.check_lu(d["A"], d["B"], w.layout, got, orc, kappa=d.get("kappa"))


@pytest.mark.parametrize("chunk", [128, 1])
def test_host_cholesky(chunk):
    d = W.make("chol_f64_n32", 1000 if chunk > 1 else 40)
    A, B = d["A"], d["B"]
    dev = parity.gpu_chol(A, B, COL_MAJOR)
    tA, tB = _pinned(A), _pinned(B)
    info = torch.full((A.shape[0],), SENT, dtype=torch.int32).pin_memory()
    bs.bs_potrf_potrs_batched_host(tA, tB, info, COL_MAJOR, bs.BS_LOWER, chunk=chunk)
    got = (tA.numpy(), tB.numpy(), info.numpy())
    for g, r in zip(got, dev):
        assert np.array_equal(g, r, equal_nan=True), chunk
    orc = oracle.potrf_potrs(A, B, COL_MAJOR, nthreads=NT)
    parity.check_chol(A, B, COL_MAJOR, got, orc)


def test_host_bdsv():
    d = W.make("bdsv_f64_32x8", 129)
    dev = parity.gpu_bdsv(d["strips"], d["x"])
    tS, tX = _pinned(d["strips"]), _pinned(d["x"])
    info = torch.full((d["strips"].shape[0],), SENT, dtype=torch.int32).pin_memory()
    bs.bs_bdsv_batched_host(tS, tX, info, chunk=40)
    got = (tS.numpy(), tX.numpy(), info.numpy())
    for g, r in zip(got, dev):
        assert np.array_equal(g, r, equal_nan=True)
    orc = oracle.bdsv(d["strips"], d["x"], nthreads=NT)
    parity.check_bdsv(d["strips"], d["x"], got, orc)


def test_host_plan_reuse_and_one_stream():
    """A plan (workspace and streams) serves several calls; both streams the same stream
    is correct too (no overlap)."""
    d = W.make("lu_f32_n16", 777)
    w = d["workload"]
    dev = parity.gpu_lu(d["A"], d["B"], w.layout)
    s = torch.cuda.Stream()
    plan = bs.getrf_getrs_host_plan(bs.BS_FP32, 16, 4, 64, streams=(s, s))
    for _ in range(2):
        tA, tB = _pinned(d["A"]), _pinned(d["B"])
        ipiv = torch.zeros((777, 16), dtype=torch.int32).pin_memory()
        info = torch.zeros(777, dtype=torch.int32).pin_memory()
        bs.bs_getrf_getrs_batched_host(tA, tB, ipiv, info, w.layout, chunk=64, plan=plan)
        for g, r in zip((tA.numpy(), tB.numpy(), ipiv.numpy(), info.numpy()), dev):
            assert np.array_equal(g, r)
