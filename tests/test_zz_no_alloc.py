"""bs_getrf_getrs_batched_host_static: the host-resident LU on the library's own static
device scratch (no workspace argument, no allocation). Its results must equal the device
call's bit for bit; the chunk shrinks until two slots fit the scratch; back-to-back calls
on the same two streams stay ordered."""
import numpy as np
import pytest
import torch

import dense_linear_solvers_gb300 as bs
from dense_linear_solvers_gb300 import _build
from gen import workloads as W
from tests import parity

FAKE = 0x10000  # never dereferenced: every host-side call below returns before any copy


def test_static_entry_point_argument_errors():
    _build.build()
    L = bs.lib()
    f = L.bs_getrf_getrs_batched_host_static
    A, B, P, I = FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000
    assert f(bs.BS_FP32, 0, 16, 4, 0, None, None, None, None, 16, None, None) == bs.BS_OK
    assert f(bs.BS_FP32, 0, 16, 4, 5, A, B, P, I, 0, None, None) == bs.BS_ERR_INVALID_ARG
    assert f(bs.BS_FP32, 0, 129, 4, 5, A, B, P, I, 16, None, None) == bs.BS_ERR_UNSUPPORTED
    assert f(bs.BS_FP64, 1, 16, -2, 5, A, B, P, I, 16, None, None) == bs.BS_ERR_INVALID_ARG


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def _static(A, B, layout, chunk, streams=None):
    tA, tB = _pinned(A), _pinned(B)
    ipiv = torch.full((A.shape[0], A.shape[1]), parity.SENTINEL, dtype=torch.int32).pin_memory()
    info = torch.full((A.shape[0],), parity.SENTINEL, dtype=torch.int32).pin_memory()
    bs.bs_getrf_getrs_batched_host_static(tA, tB, ipiv, info, layout, chunk=chunk,
                                          streams=streams)
    return tA.numpy(), tB.numpy(), ipiv.numpy(), info.numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("name,batch,chunk", [
    ("lu_f32_n16", None, 16384), ("lu_f32_n16", 1037, 100), ("lu_f64_n64", 300, 16384),
])
def test_static_scratch_matches_device_call(name, batch, chunk):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = W.make(name, batch)
    w = d["workload"]
    dev = parity.gpu_lu(d["A"], d["B"], w.layout)
    got = _static(d["A"], d["B"], w.layout, chunk)
    for g, r in zip(got, dev):
        assert np.array_equal(g, r), (name, batch, chunk)


@pytest.mark.gpu
def test_static_scratch_chunk_shrinks_for_large_systems():
    """FP64 n=128 nrhs=8: a system takes about 140 KB, so a requested chunk of 16384 is
    halved to 128 before two slots fit 64 MiB; three chunks for 300 systems."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rng = np.random.default_rng(3030)
    A = rng.standard_normal((300, 128, 128))
    B = rng.standard_normal((300, 128, 8))
    dev = parity.gpu_lu(A, B, W.ROW_MAJOR)
    got = _static(A, B, W.ROW_MAJOR, 16384)
    for g, r in zip(got, dev):
        assert np.array_equal(g, r)


@pytest.mark.gpu
def test_static_scratch_back_to_back_on_the_same_streams():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = W.make("lu_f32_n16", 5000)
    w = d["workload"]
    dev = parity.gpu_lu(d["A"], d["B"], w.layout)
    streams = (torch.cuda.Stream(), torch.cuda.Stream())
    outs = []
    for _ in range(2):
        tA, tB = _pinned(d["A"]), _pinned(d["B"])
        ipiv = torch.zeros((5000, 16), dtype=torch.int32).pin_memory()
        info = torch.zeros(5000, dtype=torch.int32).pin_memory()
        bs.bs_getrf_getrs_batched_host_static(tA, tB, ipiv, info, w.layout, chunk=1024,
                                              streams=streams, sync=False)
        outs.append((tA, tB, ipiv, info))
    for s in streams:
        s.synchronize()
    for o in outs:
        for g, r in zip(o, dev):
            assert np.array_equal(g.numpy(), r)


@pytest.mark.gpu
def test_static_scratch_calls_of_different_shapes_on_the_same_streams():
    """A call with small chunks, then without a sync a call whose chunk slot is far
    larger, both queued on the same two streams in the same order: the fixed slot offsets
    keep the second call from overwriting what the first still reads."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    small = W.make("lu_f32_n16", 6000)
    rng = np.random.default_rng(4040)
    A64 = rng.standard_normal((700, 64, 64))
    B64 = rng.standard_normal((700, 64, 8))
    dev_small = parity.gpu_lu(small["A"], small["B"], small["workload"].layout)
    dev_large = parity.gpu_lu(A64, B64, W.ROW_MAJOR)
    streams = (torch.cuda.Stream(), torch.cuda.Stream())
    calls = [(small["A"], small["B"], small["workload"].layout, 512),
             (A64, B64, W.ROW_MAJOR, 256)]
    outs = []
    for A, B, layout, chunk in calls:
        tA, tB = _pinned(A), _pinned(B)
        ipiv = torch.zeros(A.shape[:2], dtype=torch.int32).pin_memory()
        info = torch.zeros(A.shape[0], dtype=torch.int32).pin_memory()
        bs.bs_getrf_getrs_batched_host_static(tA, tB, ipiv, info, layout, chunk=chunk,
                                              streams=streams, sync=False)
        outs.append((tA, tB, ipiv, info))
    for s in streams:
        s.synchronize()
    for o, dev in zip(outs, (dev_small, dev_large)):
        for g, r in zip(o, dev):
            assert np.array_equal(g.numpy(), r)
