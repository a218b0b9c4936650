"""Seeded synthetic inputs for the batched small dense solvers.

This module is shared by the tests, the benchmark and the smoke check. It holds none
of the solvers' arithmetic: it only draws random matrices with the shapes, value
distributions and structure of the five workloads below, and lays them out in memory.

Determinism: every workload draws from NumPy ``default_rng`` streams keyed by
``[seed, stream, chunk]`` with chunks of CHUNK systems, one stream per quantity. The
first m systems of a batch are therefore the same whatever the batch size, so a small
test batch is a prefix of the full-size one.

Storage convention: matrices are returned as raw storage arrays. A row-major n x n
matrix is stored as ``M`` (shape (batch, n, n)); a column-major one as ``M^T`` (the
memory lists columns). B (n x nrhs) follows A's layout: shape (batch, n, nrhs)
row-major, (batch, nrhs, n) column-major.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

ROW_MAJOR = 0
COL_MAJOR = 1
SEED_BASE = 20261202
CHUNK = 4096


@dataclass(frozen=True)
class Workload:
    name: str
    op: str            # "getrf_getrs" | "potrf_potrs" | "bdsv"
    dtype: type
    n: int             # matrix order (bdsv: block size)
    nrhs: int          # right-hand sides (bdsv: 1)
    batch: int
    layout: int        # ROW_MAJOR / COL_MAJOR (bdsv: strips are row-major)
    seed: int
    nbr: int = 0       # bdsv: number of block rows
    text: str = ""
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "lu_f64_n8": Workload(
        "lu_f64_n8", "getrf_getrs", np.float64, 8, 1, 1024, ROW_MAJOR, SEED_BASE + 0,
        text="LU FP64 n=8 nrhs=1 batch=1024 row-major; A, b iid U[-1,1]; systems 0..15 "
             "have column (i mod 8) zeroed"),
    "lu_f32_n16": Workload(
        "lu_f32_n16", "getrf_getrs", np.float32, 16, 4, 65536, ROW_MAJOR, SEED_BASE + 1,
        text="LU FP32 n=16 nrhs=4 batch=65536 row-major; A, B iid N(0,1)"),
    "chol_f64_n32": Workload(
        "chol_f64_n32", "potrf_potrs", np.float64, 32, 1, 262144, COL_MAJOR, SEED_BASE + 2,
        text="Cholesky FP64 n=32 nrhs=1 batch=262144 column-major lower; A = G G^T + 32 I, "
             "G iid N(0,1); b iid N(0,1); 1% of systems get A[k][k] = -1"),
    "lu_f64_n64": Workload(
        "lu_f64_n64", "getrf_getrs", np.float64, 64, 8, 65536, ROW_MAJOR, SEED_BASE + 3,
        text="LU FP64 n=64 nrhs=8 batch=65536 row-major; A = U diag(s) V^T, U, V Haar, "
             "kappa log-uniform in [1e2, 1e8], s log-spaced 1..1/kappa; B iid U[-1,1]"),
    "bdsv_f64_32x8": Workload(
        "bdsv_f64_32x8", "bdsv", np.float64, 8, 1, 16384, ROW_MAJOR, SEED_BASE + 4, nbr=32,
        text="bdsv FP64 NBR=32 BS=8 batch=16384; C_i iid U[-0.5,0.5]/8, R_i = C_i, "
             "L_{i+1} = C_i^T; D_i = M_i M_i^T + 10 I, M_i iid N(0,1)/sqrt(8); b iid N(0,1)"),
}


# Inputs of rows measured beside the five workloads (not configurations of their own):
# Cholesky beyond one CTA, with the recipe of chol_f64_n32 at a larger order.
EXTRA_WORKLOADS = {
    "chol_f64_n256": Workload(
        "chol_f64_n256", "potrf_potrs", np.float64, 256, 1, 2048, COL_MAJOR, SEED_BASE + 5,
        text="Cholesky FP64 n=256 nrhs=1 batch=2048 column-major lower; A = G G^T + 256 I, "
             "G iid N(0,1); b iid N(0,1); 1% of systems get A[k][k] = -1"),
}


def workload(name: str) -> Workload:
    """One of WORKLOADS or EXTRA_WORKLOADS by name."""
    return WORKLOADS[name] if name in WORKLOADS else EXTRA_WORKLOADS[name]


def _rng(seed: int, stream: int, chunk: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream, chunk])


def _chunks(batch: int):
    for c in range(0, (batch + CHUNK - 1) // CHUNK):
        lo = c * CHUNK
        yield c, lo, min(batch, lo + CHUNK)


def to_storage(M: np.ndarray, layout: int) -> np.ndarray:
    """Logical (batch, r, c) matrices -> raw storage in the given layout."""
    return np.ascontiguousarray(M if layout == ROW_MAJOR else np.swapaxes(M, 1, 2))


def from_storage(S: np.ndarray, layout: int) -> np.ndarray:
    """Raw storage -> logical (batch, r, c) matrices (a view for row-major)."""
    return S if layout == ROW_MAJOR else np.swapaxes(S, 1, 2)


def interleave(S: np.ndarray, w: int) -> np.ndarray:
    """Per-system storage (batch, ...) -> the flat interleaved batched layout with w
    systems per block: element e of system s at (s // w) * w * size + e * w + s % w
    (w = 1: the systems one after another; w >= batch: SoA). Slots of the last block
    past the batch hold NaN, so that a stray read shows."""
    batch = S.shape[0]
    size = int(np.prod(S.shape[1:], dtype=np.int64))
    nb = -(-batch // w)
    fill = np.nan if np.issubdtype(S.dtype, np.floating) else -7
    P = np.full((nb * w, size), fill, dtype=S.dtype)
    P[:batch] = S.reshape(batch, size)
    return np.ascontiguousarray(P.reshape(nb, w, size).transpose(0, 2, 1)).reshape(-1)


def deinterleave(flat: np.ndarray, batch: int, w: int, shape) -> np.ndarray:
    """Inverse of interleave: the flat interleaved array -> (batch, *shape)."""
    size = int(np.prod(shape, dtype=np.int64))
    nb = -(-batch // w)
    P = flat[:nb * w * size].reshape(nb, size, w).transpose(0, 2, 1).reshape(nb * w, size)
    return np.ascontiguousarray(P[:batch]).reshape((batch,) + tuple(shape))


def _bmm(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    # Batched matrix product through torch's CPU BLAS binding (NumPy's stacked matmul
    # is slow for many tiny matrices); the inputs are the generator's own draws.
    import torch
    return torch.bmm(torch.from_numpy(np.ascontiguousarray(a)),
                     torch.from_numpy(np.ascontiguousarray(b))).numpy()


def _haar(rng: np.random.Generator, m: int, n: int) -> np.ndarray:
    # Haar-distributed orthogonal matrices: QR of a Gaussian matrix with the signs of
    # R's diagonal moved into Q (Mezzadri, "How to generate random matrices from the
    # classical compact groups", 2007). The batched QR runs through torch's CPU LAPACK
    # binding, which spreads the independent factorizations over the host cores.
    Z = rng.standard_normal((m, n, n))
    import torch
    Qt, Rt = torch.linalg.qr(torch.from_numpy(Z))
    Q, R = Qt.numpy(), Rt.numpy()
    d = np.sign(np.diagonal(R, axis1=1, axis2=2))
    d[d == 0] = 1.0
    return Q * d[:, None, :]


def make(name: str, batch: int | None = None) -> dict:
    """Inputs of one workload as raw storage arrays, plus metadata.

    Returns a dict with "A", "B" (LU/Cholesky) or "strips", "x" (bdsv), and for
    workloads with planted failures the expected info codes of the planted systems.
    """
    w = workload(name)
    batch = w.batch if batch is None else int(batch)
    if w.op == "bdsv":
        return _make_bdsv(w, batch)
    n, nrhs, dt = w.n, w.nrhs, w.dtype
    A = np.empty((batch, n, n), dt)
    B = np.empty((batch, n, nrhs), dt)
    planted = {}
    for c, lo, hi in _chunks(batch):
        m = hi - lo
        if name == "lu_f64_n8":
            A[lo:hi] = _rng(w.seed, 0, c).uniform(-1.0, 1.0, (m, n, n))
            B[lo:hi] = _rng(w.seed, 1, c).uniform(-1.0, 1.0, (m, n, nrhs))
        elif name == "lu_f32_n16":
            A[lo:hi] = _rng(w.seed, 0, c).standard_normal((m, n, n), dtype=np.float32)
            B[lo:hi] = _rng(w.seed, 1, c).standard_normal((m, n, nrhs), dtype=np.float32)
        elif name in ("chol_f64_n32", "chol_f64_n256"):
            G = _rng(w.seed, 0, c).standard_normal((m, n, n))
            A[lo:hi] = _bmm(G, np.swapaxes(G, 1, 2)) + n * np.eye(n)
            B[lo:hi] = _rng(w.seed, 1, c).standard_normal((m, n, nrhs))
            sel = _rng(w.seed, 2, c).random((m, 2))
            for i in np.nonzero(sel[:, 0] < 0.01)[0]:
                k = int(sel[i, 1] * n)
                A[lo + i, k, k] = -1.0
                planted[lo + int(i)] = k + 1
        elif name == "lu_f64_n64":
            U = _haar(_rng(w.seed, 0, c), m, n)
            V = _haar(_rng(w.seed, 1, c), m, n)
            logk = _rng(w.seed, 2, c).uniform(2.0, 8.0, m)
            sig = 10.0 ** (-np.linspace(0.0, 1.0, n)[None, :] * logk[:, None])
            A[lo:hi] = _bmm(U * sig[:, None, :], np.swapaxes(V, 1, 2))
            B[lo:hi] = _rng(w.seed, 3, c).uniform(-1.0, 1.0, (m, n, nrhs))
        else:
            raise KeyError(name)
    if name == "lu_f64_n8":
        for i in range(min(16, batch)):
            A[i, :, i % n] = 0.0
            planted[i] = (i % n) + 1
    out = {"A": to_storage(A, w.layout), "B": to_storage(B, w.layout), "planted_info": planted,
           "workload": w, "batch": batch}
    if name == "lu_f64_n64":
        out["kappa"] = np.concatenate(
            [10.0 ** _rng(w.seed, 2, c).uniform(2.0, 8.0, hi - lo) for c, lo, hi in _chunks(batch)])
    return out


def _make_bdsv(w: Workload, batch: int) -> dict:
    nbr, bs, dt = w.nbr, w.n, w.dtype
    strips = np.zeros((batch, nbr, bs, 3 * bs), dt)
    xpad = np.zeros((batch, (nbr + 2) * bs), dt)
    for c, lo, hi in _chunks(batch):
        m = hi - lo
        C = _rng(w.seed, 0, c).uniform(-0.5, 0.5, (m, nbr - 1, bs, bs)) / 8.0
        M = _rng(w.seed, 1, c).standard_normal((m, nbr, bs, bs)) / np.sqrt(8.0)
        MMt = _bmm(M.reshape(-1, bs, bs), np.swapaxes(M, 2, 3).reshape(-1, bs, bs))
        D = MMt.reshape(M.shape) + 10.0 * np.eye(bs)
        strips[lo:hi, :, :, bs:2 * bs] = D
        strips[lo:hi, :nbr - 1, :, 2 * bs:] = C                       # R_i = C_i
        strips[lo:hi, 1:, :, :bs] = np.swapaxes(C, 2, 3)             # L_{i+1} = C_i^T
        xpad[lo:hi, bs:(nbr + 1) * bs] = _rng(w.seed, 2, c).standard_normal((m, nbr * bs))
    return {"strips": strips, "x": xpad, "planted_info": {}, "workload": w, "batch": batch}


def assemble_bdsv_dense(strips: np.ndarray) -> np.ndarray:
    """Dense (batch, nbr*bs, nbr*bs) matrices from [L|D|R] strips (test helper)."""
    batch, nbr, bs = strips.shape[0], strips.shape[1], strips.shape[2]
    N = nbr * bs
    Adense = np.zeros((batch, N, N), strips.dtype)
    for br in range(nbr):
        r0 = br * bs
        Adense[:, r0:r0 + bs, r0:r0 + bs] = strips[:, br, :, bs:2 * bs]
        if br > 0:
            Adense[:, r0:r0 + bs, r0 - bs:r0] = strips[:, br, :, :bs]
        if br < nbr - 1:
            Adense[:, r0:r0 + bs, r0 + bs:r0 + 2 * bs] = strips[:, br, :, 2 * bs:]
    return Adense
