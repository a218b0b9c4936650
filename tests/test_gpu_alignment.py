"""Operands that are 16-byte aligned but not 32-byte aligned (the C ABI's requirement is
16 bytes): the kernels that move rows in 32-byte pieces when the base allows take their
16-byte paths there, with the same results bit for bit, equal to the oracle's."""
import numpy as np
import pytest
import torch

import dense_linear_solvers_gb300 as bs
import oracle
from gen.workloads import ROW_MAJOR
from tests import parity

pytestmark = pytest.mark.gpu
SENT = parity.SENTINEL


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bs.lib()


def _placed(a: np.ndarray, offset_bytes: int):
    """A device copy of a whose first element sits offset_bytes past a 256-byte boundary."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    pad = offset_bytes // t.element_size()
    buf = torch.empty(t.numel() + pad, dtype=t.dtype, device="cuda")
    view = buf[pad:pad + t.numel()].view(t.shape)
    view.copy_(t.to("cuda"))
    assert view.data_ptr() % 256 == offset_bytes
    return view


@pytest.mark.parametrize("n", [16, 12])
@pytest.mark.parametrize("nrhs", [0, 1, 3, 4, 8])
def test_lu_rows_off_32_bytes(n, nrhs):
    rng = np.random.default_rng(3131 + 10 * n + nrhs)
    batch = 77
    A = rng.standard_normal((batch, n, n)).astype(np.float32)
    A[3, :, 2] = 0                       # a singular system
    B = rng.standard_normal((batch, n, max(nrhs, 1))).astype(np.float32)
    outs = []
    for off in (0, 16):
        tA = _placed(A, off)
        ipiv = torch.full((batch, n), SENT, dtype=torch.int32, device="cuda")
        info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
        if nrhs == 0:
            bs.bs_getrf_batched(tA, ipiv, info, ROW_MAJOR)
            tB = None
        else:
            tB = _placed(B, off)
            bs.bs_getrf_getrs_batched(tA, tB, ipiv, info, ROW_MAJOR)
        torch.cuda.synchronize()
        outs.append([tA.cpu().numpy(), None if tB is None else tB.cpu().numpy(),
                     ipiv.cpu().numpy(), info.cpu().numpy()])
    for x, y in zip(outs[0], outs[1]):
        if x is not None:
            assert np.array_equal(x, y)
    if nrhs == 0:
        Fo, ipo, info_o, tie = oracle.getrf(A, ROW_MAJOR)
        clean = tie < 0
        assert np.array_equal(outs[1][0][clean], Fo[clean])
    else:
        Fo, Xo, ipo, info_o, tie = oracle.getrf_getrs(A, B, ROW_MAJOR)
        clean = tie < 0
        assert np.array_equal(outs[1][0][clean], Fo[clean])
        assert np.array_equal(outs[1][1][clean], Xo[clean])
    assert np.array_equal(outs[1][2][clean], ipo[clean])
    assert np.array_equal(outs[1][3], info_o) and outs[1][3][3] > 0


def _bdsv_case(rng, dtype, batch, nbr, bsz):
    strips = np.zeros((batch, nbr, bsz, 3 * bsz))
    C = rng.uniform(-0.5, 0.5, (batch, nbr - 1, bsz, bsz)) / bsz
    M = rng.standard_normal((batch, nbr, bsz, bsz)) / np.sqrt(bsz)
    strips[:, :, :, bsz:2 * bsz] = M @ np.swapaxes(M, 2, 3) + 4.0 * np.eye(bsz)
    strips[:, :nbr - 1, :, 2 * bsz:] = C
    strips[:, 1:, :, :bsz] = np.swapaxes(C, 2, 3)
    xpad = np.zeros((batch, (nbr + 2) * bsz))
    xpad[:, bsz:(nbr + 1) * bsz] = rng.standard_normal((batch, nbr * bsz))
    strips[7, nbr // 2, 0, bsz] = -1.0      # an indefinite knot inside the sweep
    return strips.astype(dtype), xpad.astype(dtype)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("bsz", [4, 8])
def test_bdsv_off_32_bytes(dtype, bsz):
    """Fused sweep, factor alone and solve alone, strips and x 16 bytes past a 32-byte
    boundary, against the aligned calls and the oracle."""
    rng = np.random.default_rng(3232 + bsz)
    batch, nbr = 45, 9
    strips, xpad = _bdsv_case(rng, dtype, batch, nbr, bsz)
    res = []
    for off in (0, 16):
        tS, tX = _placed(strips, off), _placed(xpad, off)
        info = torch.full((batch,), SENT, dtype=torch.int32, device="cuda")
        bs.bs_bdsv_batched(tS, tX, info)
        fS, fI = _placed(strips, off), torch.full((batch,), SENT, dtype=torch.int32,
                                                  device="cuda")
        bs.bs_bdsv_factor_batched(fS, fI)
        sX = _placed(xpad, off)
        bs.bs_bdsv_solve_batched(fS, sX)
        torch.cuda.synchronize()
        res.append([x.cpu().numpy() for x in (tS, tX, info, fS, fI, sX)])
    for x, y in zip(res[0], res[1]):
        assert np.array_equal(x, y, equal_nan=True)
    So, Xo, info_o = oracle.bdsv(strips, xpad)
    S1, X1, I1, F1, FI1, SX1 = res[1]
    assert np.array_equal(I1, info_o) and I1[7] > 0 and np.array_equal(FI1, info_o)
    ok = info_o == 0
    assert np.array_equal(X1[ok], Xo[ok])
    assert np.array_equal(SX1[ok], Xo[ok])
    assert np.array_equal(F1[ok], S1[ok])
