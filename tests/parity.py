"""GPU-vs-oracle parity checks (test-only helpers).

The criteria (per system):
  * info bit-exact; pivots bit-exact, except from the first step whose two largest
    candidates the oracle found within 1e-6 relative of each other (a near tie);
  * systems that fail (info != 0) return X = 0;
  * normwise backward error ||A x - b|| / (||A|| ||x|| + ||b||) <= 8 n eps(dtype)
    (infinity norms, residual in double-double), for every system that succeeded;
  * forward error ||x - x_oracle|| / ||x_oracle|| <= 1e-4 (FP32) / 1e-10 (FP64) on
    systems with condition number <= 1e4.
"""
from __future__ import annotations

import numpy as np
import torch

import dense_linear_solvers_gb300 as bs
from gen.workloads import COL_MAJOR, ROW_MAJOR, from_storage
from tests.numerics import backward_error, eps_of, forward_error

FWD_TOL = {np.dtype(np.float32): 1e-4, np.dtype(np.float64): 1e-10}
SENTINEL = -7


def gpu_lu(A, B, layout):
    dev = torch.device("cuda")
    tA = torch.from_numpy(np.ascontiguousarray(A)).to(dev)
    tB = torch.from_numpy(np.ascontiguousarray(B)).to(dev)
    batch, n = A.shape[0], A.shape[1]
    ipiv = torch.full((batch, n), SENTINEL, dtype=torch.int32, device=dev)
    info = torch.full((batch,), SENTINEL, dtype=torch.int32, device=dev)
    bs.bs_getrf_getrs_batched(tA, tB, ipiv, info, layout)
    torch.cuda.synchronize()
    return tA.cpu().numpy(), tB.cpu().numpy(), ipiv.cpu().numpy(), info.cpu().numpy()


def gpu_chol(A, B, layout):
    dev = torch.device("cuda")
    tA = torch.from_numpy(np.ascontiguousarray(A)).to(dev)
    tB = torch.from_numpy(np.ascontiguousarray(B)).to(dev)
    info = torch.full((A.shape[0],), SENTINEL, dtype=torch.int32, device=dev)
    bs.bs_potrf_potrs_batched(tA, tB, info, layout, bs.BS_LOWER)
    torch.cuda.synchronize()
    return tA.cpu().numpy(), tB.cpu().numpy(), info.cpu().numpy()


def gpu_bdsv(strips, xpad):
    dev = torch.device("cuda")
    tS = torch.from_numpy(np.ascontiguousarray(strips)).to(dev)
    tX = torch.from_numpy(np.ascontiguousarray(xpad)).to(dev)
    info = torch.full((strips.shape[0],), SENTINEL, dtype=torch.int32, device=dev)
    bs.bs_bdsv_batched(tS, tX, info)
    torch.cuda.synchronize()
    return tS.cpu().numpy(), tX.cpu().numpy(), info.cpu().numpy()


def condition_numbers(A_logical):
    s = np.linalg.svd(np.asarray(A_logical, np.float64), compute_uv=False)
    with np.errstate(divide="ignore", invalid="ignore"):   # a zero matrix: 0 / 0
        return np.where(s[:, -1] > 0, s[:, 0] / s[:, -1], np.inf)


def _x_logical(X, layout):
    return from_storage(X, layout)


class Report(dict):
    """Counts of what was compared, kept for the test log."""


def check_lu(A, B, layout, gpu, orc, kappa=None):
    LUg, Xg, ipg, infg = gpu
    LUo, Xo, ipo, info_o, tie = orc
    dt = np.dtype(A.dtype)
    n = A.shape[1]
    eps = eps_of(dt)
    rep = Report(systems=A.shape[0])
    assert np.all(infg != SENTINEL) and np.all(ipg != SENTINEL), "outputs left unwritten"
    clean = tie < 0
    # info: exact where the oracle met no near tie before its first failing step
    info_cmp = clean | ((info_o > 0) & (info_o - 1 < tie))
    bad = np.nonzero(info_cmp & (infg != info_o))[0]
    assert bad.size == 0, f"info differs on systems {bad[:10]}: gpu {infg[bad[:10]]} oracle {info_o[bad[:10]]}"
    # pivots: exact on every step before the first near tie
    steps = np.where(clean, n, tie)
    mask = np.arange(n)[None, :] < steps[:, None]
    bad = np.nonzero(np.any(mask & (ipg != ipo), axis=1))[0]
    assert bad.size == 0, f"ipiv differs on systems {bad[:10]}"
    rep["near_tie_systems"] = int((~clean).sum())
    # failed systems: X = 0
    Xl = _x_logical(Xg, layout)
    failed = infg != 0
    assert np.all(Xl[failed] == 0)
    rep["failed_systems"] = int(failed.sum())
    # backward error on the systems that succeeded
    Al = from_storage(A, layout)
    Bl = _x_logical(B, layout)
    okm = ~failed
    if okm.any():
        be = backward_error(Al[okm], Xl[okm], Bl[okm])
        worst = float(be.max())
        assert worst <= 8 * n * eps, f"backward error {worst:.3e} > {8 * n * eps:.3e}"
        rep["max_backward_error"] = worst
    # forward error on kappa <= 1e4
    if kappa is None:
        kappa = condition_numbers(Al)
    fm = okm & (info_o == 0) & (kappa <= 1e4)
    if fm.any():
        fe = forward_error(Xl[fm], _x_logical(Xo, layout)[fm])
        worst = float(fe.max())
        assert worst <= FWD_TOL[dt], f"forward error {worst:.3e} > {FWD_TOL[dt]:.0e}"
        rep["max_forward_error"] = worst
        rep["forward_checked"] = int(fm.sum())
    # the kernels perform the oracle's operations in the oracle's order: where the pivots
    # agree (no near tie) and the factorization succeeded, L\U and X are equal bit for bit
    same = okm & clean & (info_o == 0)
    eq = (np.all((LUg[same] == LUo[same]).reshape(same.sum(), -1), axis=1)
          & np.all((Xg[same] == Xo[same]).reshape(same.sum(), -1), axis=1))
    bad = np.nonzero(same)[0][~eq]
    assert bad.size == 0, f"L\\U or X not bitwise equal to the oracle on systems {bad[:10]}"
    rep["bitwise_equal_systems"] = int(eq.sum())
    rep["compared_for_bitwise"] = int(same.sum())
    return rep


def check_chol(A, B, layout, gpu, orc):
    Lg, Xg, infg = gpu
    Lo, Xo, info_o = orc
    dt = np.dtype(A.dtype)
    n = A.shape[1]
    eps = eps_of(dt)
    rep = Report(systems=A.shape[0])
    assert np.all(infg != SENTINEL)
    bad = np.nonzero(infg != info_o)[0]
    assert bad.size == 0, f"info differs on systems {bad[:10]}: gpu {infg[bad[:10]]} oracle {info_o[bad[:10]]}"
    # the strict upper triangle is untouched
    Al = from_storage(A, layout)
    Lgl = from_storage(Lg, layout)
    iu = np.triu_indices(n, 1)
    assert np.array_equal(Lgl[:, iu[0], iu[1]], Al[:, iu[0], iu[1]]), "upper triangle written"
    Xl = _x_logical(Xg, layout)
    failed = infg != 0
    assert np.all(Xl[failed] == 0)
    rep["failed_systems"] = int(failed.sum())
    okm = ~failed
    if okm.any():
        # the matrix the solve is judged against: the lower triangle, mirrored
        As = np.tril(Al[okm]) + np.swapaxes(np.tril(Al[okm], -1), 1, 2)
        be = backward_error(As, Xl[okm], _x_logical(B, layout)[okm])
        worst = float(be.max())
        assert worst <= 8 * n * eps, f"backward error {worst:.3e} > {8 * n * eps:.3e}"
        rep["max_backward_error"] = worst
        kappa = condition_numbers(As)
        fm = kappa <= 1e4
        if fm.any():
            fe = forward_error(Xl[okm][fm], _x_logical(Xo, layout)[okm][fm])
            worst = float(fe.max())
            assert worst <= FWD_TOL[dt], f"forward error {worst:.3e}"
            rep["max_forward_error"] = worst
        Lol = from_storage(Lo, layout)
        il = np.tril_indices(n)
        diff = np.abs(Lgl[okm][:, il[0], il[1]] - Lol[okm][:, il[0], il[1]]).max()
        assert diff <= 64 * n * eps * max(np.abs(Lol[okm][:, il[0], il[1]]).max(), 1.0)
        rep["bitwise_equal_systems"] = int(np.sum(np.all(
            (Lgl[okm][:, il[0], il[1]] == Lol[okm][:, il[0], il[1]]), axis=1)))
    return rep


def bdsv_backward_error(strips, b_pad, x_pad):
    """Block-row residual r_k = b_k - [L|D|R] [x_{k-1}; x_k; x_{k+1}] (GLASS's bdmv
    window over the padded vector), normalized as the dense backward error."""
    batch, nbr, bs_ = strips.shape[0], strips.shape[1], strips.shape[2]
    from tests.numerics import residual_dd
    strips = np.array(strips, np.float64)
    strips[:, 0, :, :bs_] = 0.0            # L_0 and R_{nbr-1} are not part of the matrix
    strips[:, nbr - 1, :, 2 * bs_:] = 0.0
    x_pad = np.array(x_pad, np.float64)
    x_pad[:, :bs_] = 0.0                   # the matvec window reads zero pads
    x_pad[:, (nbr + 1) * bs_:] = 0.0
    Ablk = strips.reshape(batch * nbr, bs_, 3 * bs_)
    win = np.stack([x_pad[:, br * bs_: br * bs_ + 3 * bs_] for br in range(nbr)], axis=1)
    Xw = win.reshape(batch * nbr, 3 * bs_, 1).astype(np.float64)
    Bb = b_pad[:, bs_:(nbr + 1) * bs_].reshape(batch * nbr, bs_, 1).astype(np.float64)
    R = residual_dd(Ablk, Xw, Bb).reshape(batch, nbr * bs_)
    an = np.abs(Ablk).sum(axis=2).reshape(batch, nbr * bs_).max(axis=1)
    xn = np.abs(x_pad[:, bs_:(nbr + 1) * bs_]).max(axis=1)
    bn = np.abs(b_pad[:, bs_:(nbr + 1) * bs_]).max(axis=1)
    return np.abs(R).max(axis=1) / (an * xn + bn)


def check_bdsv(strips, xpad, gpu, orc):
    Sg, Xg, infg = gpu
    So, Xo, info_o = orc
    dt = np.dtype(strips.dtype)
    eps = eps_of(dt)
    batch, nbr, bs_ = strips.shape[0], strips.shape[1], strips.shape[2]
    N = nbr * bs_
    rep = Report(systems=batch)
    assert np.all(infg != SENTINEL)
    bad = np.nonzero(infg != info_o)[0]
    assert bad.size == 0, f"info differs on systems {bad[:10]}"
    # pads and RIGHT slots untouched
    assert np.array_equal(Xg[:, :bs_], xpad[:, :bs_]) and np.array_equal(Xg[:, N + bs_:], xpad[:, N + bs_:])
    assert np.array_equal(Sg[:, :, :, 2 * bs_:], strips[:, :, :, 2 * bs_:])
    failed = infg != 0
    assert np.all(Xg[failed][:, bs_:bs_ + N] == 0)
    okm = ~failed
    if okm.any():
        iu = np.triu_indices(bs_, 1)
        main_g = Sg[okm][:, :, :, bs_:2 * bs_]
        assert np.array_equal(main_g[:, :, iu[0], iu[1]],
                              strips[okm][:, :, :, bs_:2 * bs_][:, :, iu[0], iu[1]])
        be = bdsv_backward_error(strips[okm], xpad[okm], Xg[okm])
        worst = float(be.max())
        assert worst <= 8 * N * eps, f"backward error {worst:.3e} > {8 * N * eps:.3e}"
        rep["max_backward_error"] = worst
        fe = forward_error(Xg[okm][:, bs_:bs_ + N], Xo[okm][:, bs_:bs_ + N])
        worst = float(fe.max())
        assert worst <= FWD_TOL[dt], f"forward error {worst:.3e}"
        rep["max_forward_error"] = worst
        tol = 64 * N * eps
        assert np.abs(Sg[okm] - So[okm]).max() <= tol * max(np.abs(So[okm]).max(), 1.0)
        rep["bitwise_equal_systems"] = int(np.sum(np.all(
            (Sg[okm] == So[okm]).reshape(okm.sum(), -1), axis=1)
            & np.all(Xg[okm] == Xo[okm], axis=1)))
    return rep
