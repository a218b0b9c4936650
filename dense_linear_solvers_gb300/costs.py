"""Algorithmic bytes and flops per system, for roofline accounting.

Bytes: every element the method must touch, once in and once out; operands the method
skips are not counted (the strict upper triangle of a lower-fill Cholesky, the RIGHT
slots and L_0 of the block-tridiagonal strips, the pad blocks of its vector). Pivots
and info are int32. With ``full_matrix=True`` the Cholesky count reads and writes the
whole n x n matrix instead, the accounting of the RUDA page ("ruSOLVER: small-matrix
kernel optimisation": logical bytes per system on the success path), which this module
reproduces for FP32, n = 32, nrhs = 8 (10,244 bytes Cholesky, 10,372 bytes LU).

Flops: the standard count, a fused multiply-add is 2 flops, a division or a square root
is 1.
"""
from __future__ import annotations

HBM_FALLBACK_GBS = 6800.0          # used only when no measured figure is available
SM_COUNT = 152
SM_MAX_MHZ = 2070.0
FP64_FMA_PER_CLK_PER_SM = 2        # GB300: FP64 issues 1/64 of the FP32 lane rate
FP32_FMA_PER_CLK_PER_SM = 128


def alu_peak_tflops(dtype_size: int) -> float:
    """Peak of plain FMA arithmetic from the unit counts and the maximum SM clock."""
    per_clk = FP64_FMA_PER_CLK_PER_SM if dtype_size == 8 else FP32_FMA_PER_CLK_PER_SM
    return SM_COUNT * per_clk * 2 * SM_MAX_MHZ * 1e6 / 1e12


def getrf_getrs_bytes(n: int, nrhs: int, elem: int) -> int:
    return 2 * n * n * elem + 2 * n * nrhs * elem + 4 * n + 4


def potrf_potrs_bytes(n: int, nrhs: int, elem: int, full_matrix: bool = False) -> int:
    a = n * n if full_matrix else n * (n + 1) // 2
    return 2 * a * elem + 2 * n * nrhs * elem + 4


def bdsv_bytes(nbr: int, bs: int, elem: int) -> int:
    d_lower = nbr * bs * (bs + 1) // 2
    left = (nbr - 1) * bs * bs
    vec = nbr * bs
    return 2 * (d_lower + left + vec) * elem + 4


def getrf_getrs_flops(n: int, nrhs: int) -> int:
    getrf = n * (n - 1) // 2 + (n - 1) * n * (2 * n - 1) // 3
    getrs = nrhs * (2 * n * n - n)
    return getrf + getrs


def potrf_potrs_flops(n: int, nrhs: int) -> int:
    potrf = n + n * (n - 1) // 2 + (n - 1) * n * (n + 1) // 3
    potrs = 2 * n * n * nrhs
    return potrf + potrs


def bdsv_flops(nbr: int, bs: int) -> int:
    potrf = bs + bs * (bs - 1) // 2 + (bs - 1) * bs * (bs + 1) // 3
    trsm = bs ** 3
    syrk = bs * bs * (bs + 1)
    gemv = 2 * bs * bs
    trsv = bs * bs
    return potrf * nbr + (trsm + syrk) * (nbr - 1) + gemv * 2 * (nbr - 1) + trsv * 2 * nbr


# --- the factor / solve halves and the block-tridiagonal matvec -------------------------
def getrf_only(n: int, elem: int):
    return 2 * n * n * elem + 4 * n + 4, n * (n - 1) // 2 + (n - 1) * n * (2 * n - 1) // 3


def getrs_only(n: int, nrhs: int, elem: int):
    # reads L\U and ipiv, reads and writes B
    return n * n * elem + 4 * n + 2 * n * nrhs * elem, nrhs * (2 * n * n - n)


def potrf_only(n: int, elem: int):
    return 2 * (n * (n + 1) // 2) * elem + 4, n + n * (n - 1) // 2 + (n - 1) * n * (n + 1) // 3


def potrs_only(n: int, nrhs: int, elem: int):
    return (n * (n + 1) // 2) * elem + 2 * n * nrhs * elem, 2 * n * n * nrhs


def bdsv_factor_only(nbr: int, bs: int, elem: int):
    d_lower = nbr * bs * (bs + 1) // 2
    left = (nbr - 1) * bs * bs
    potrf = bs + bs * (bs - 1) // 2 + (bs - 1) * bs * (bs + 1) // 3
    flops = potrf * nbr + (bs ** 3 + bs * bs * (bs + 1)) * (nbr - 1)
    return 2 * (d_lower + left) * elem + 4, flops


def bdsv_solve_only(nbr: int, bs: int, elem: int):
    d_lower = nbr * bs * (bs + 1) // 2
    left = (nbr - 1) * bs * bs
    vec = nbr * bs
    return (d_lower + left) * elem + 2 * vec * elem, 2 * bs * bs * 2 * (nbr - 1) + bs * bs * 2 * nbr


def bdmv_bytes_flops(nbr: int, bs: int, elem: int):
    # every strip entry and the padded x in, the interior of y out
    strips = nbr * bs * 3 * bs
    return (strips + (nbr + 2) * bs + nbr * bs) * elem, 2 * strips


def per_system(op: str, n: int, nrhs: int, elem: int, nbr: int = 0):
    """(bytes, flops) of one system of a workload (n is the block size for the
    block-tridiagonal operations)."""
    # T: the row-major reading; il: an interleaved batched layout (the same work)
    if op in ("getrf_getrs", "getrf_getrs_T", "getrf_getrs_il"):
        return getrf_getrs_bytes(n, nrhs, elem), getrf_getrs_flops(n, nrhs)
    if op in ("potrf_potrs", "potrf_potrs_il"):
        return potrf_potrs_bytes(n, nrhs, elem), potrf_potrs_flops(n, nrhs)
    if op == "bdsv":
        return bdsv_bytes(nbr, n, elem), bdsv_flops(nbr, n)
    if op == "getrf":
        return getrf_only(n, elem)
    if op == "getrs":
        return getrs_only(n, nrhs, elem)
    if op == "potrf":
        return potrf_only(n, elem)
    if op == "potrs":
        return potrs_only(n, nrhs, elem)
    if op == "bdsv_factor":
        return bdsv_factor_only(nbr, n, elem)
    if op == "bdsv_solve":
        return bdsv_solve_only(nbr, n, elem)
    if op == "bdmv":
        return bdmv_bytes_flops(nbr, n, elem)
    raise KeyError(op)
