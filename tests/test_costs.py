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
