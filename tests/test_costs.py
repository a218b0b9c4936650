"""The byte and flop model against the figures the pages print (CPU only)."""
import json
import os

from dense_linear_solvers_gb300 import costs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_reproduces_ruda_logical_bytes():
    g = json.load(open(os.path.join(GOLDEN, "ruda_logical_bytes.json")))
    n, r = g["n"], g["nrhs"]
    assert costs.getrf_getrs_bytes(n, r, 4) == g["lu_bytes_per_system"]
    assert costs.potrf_potrs_bytes(n, r, 4, full_matrix=True) == g["cholesky_bytes_per_system"]


def test_workload_figures():
    # bytes and flops per system of the five workloads, counted by hand from the
    # operand sizes and the standard operation counts
    assert costs.per_system("getrf_getrs", 8, 1, 8) == (1188, 428)
    assert costs.per_system("getrf_getrs", 16, 4, 4) == (2628, 4584)
    assert costs.per_system("potrf_potrs", 32, 1, 8) == (8964, 13488)
    assert costs.per_system("getrf_getrs", 64, 8, 8) == (73988, 237728)
    assert costs.per_system("bdsv", 8, 1, 8, nbr=32) == (54276, 52288)


def test_flops_small_closed_forms():
    # n = 1: one division-free pivot, one multiply per right-hand side column
    assert costs.getrf_getrs_flops(1, 1) == 1
    # n = 2 getrf: 1 multiplier + 1 fma (2 flops); getrs: 2*(8-2) = 12
    assert costs.getrf_getrs_flops(2, 2) == 3 + 12
    assert costs.potrf_potrs_flops(1, 1) == 1 + 2
    assert abs(costs.alu_peak_tflops(8) - 1.2586) < 1e-3


def test_every_bench_row_has_a_cost():
    """Every operation the benchmark times has a cost model; the row-major reading and the
    interleaved layouts count the fused calls' bytes and flops (the same work)."""
    import bench
    for name, (base, op) in bench.NEXT_ROWS.items():
        w = bench.W.workload(base)
        b, f = costs.per_system(op, w.n, w.nrhs, 4 if w.dtype.__name__ == "float32" else 8,
                                w.nbr)
        assert b > 0 and f > 0, name
        assert name in bench.KERNEL_SOURCES, name
    for op, fused in (("getrf_getrs_T", "getrf_getrs"), ("getrf_getrs_il", "getrf_getrs"),
                      ("potrf_potrs_il", "potrf_potrs")):
        assert costs.per_system(op, 16, 4, 4) == costs.per_system(fused, 16, 4, 4)


def test_interleave_round_trip_and_addressing():
    """gen.workloads.interleave puts element e of system s at (s // w) * w * size + e * w
    + s % w, pads the last block with NaN, and deinterleave inverts it."""
    import numpy as np
    from gen.workloads import deinterleave, interleave
    X = np.arange(7 * 2 * 3, dtype=np.float64).reshape(7, 2, 3)
    for w in (1, 2, 3, 7, 10):
        f = interleave(X, w)
        nb = -(-7 // w)
        assert f.size == nb * w * 6
        for s in range(7):
            for e in range(6):
                assert f[(s // w) * w * 6 + e * w + s % w] == X[s].reshape(-1)[e]
        assert np.isnan(f).sum() == (nb * w - 7) * 6
        assert np.array_equal(deinterleave(f, 7, w, (2, 3)), X)
