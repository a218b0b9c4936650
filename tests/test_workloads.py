"""The input recipe (gen/workloads.py) has the properties the workloads are stated to have:
a small batch is a prefix of a larger one (across the 4096-system chunk boundary), the
planted failures carry the stated info codes under the oracle, the FP64 n=64 systems have
the stated singular values and the returned kappa is their 2-norm condition number, and
the block-tridiagonal systems are symmetric positive definite with the stated margin."""
import numpy as np
import pytest

import oracle
from gen import workloads as W
from gen.workloads import COL_MAJOR, ROW_MAJOR, from_storage

NT = 4


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_small_batch_is_a_prefix(name):
    small, large = W.make(name, 4100), W.make(name, 4300)
    keys = ("strips", "x") if W.WORKLOADS[name].op == "bdsv" else ("A", "B")
    for k in keys:
        assert np.array_equal(small[k], large[k][:4100]), (name, k)
        assert np.array_equal(small[k], W.make(name, 4100)[k]), (name, k)   # seeded
    assert {s: c for s, c in large["planted_info"].items() if s < 4100} == small["planted_info"]


def test_dtypes_shapes_and_storage_orders():
    for name, w in W.WORKLOADS.items():
        d = W.make(name, 10)
        if w.op == "bdsv":
            assert d["strips"].shape == (10, w.nbr, w.n, 3 * w.n)
            assert d["x"].shape == (10, (w.nbr + 2) * w.n)
            assert d["strips"].dtype == w.dtype and d["x"].dtype == w.dtype
            continue
        assert d["A"].shape == (10, w.n, w.n) and d["A"].dtype == w.dtype
        want_b = (10, w.n, w.nrhs) if w.layout == ROW_MAJOR else (10, w.nrhs, w.n)
        assert d["B"].shape == want_b and d["B"].dtype == w.dtype


def test_lu_f64_n8_zeroed_columns_give_their_info():
    d = W.make("lu_f64_n8")
    A = from_storage(d["A"], ROW_MAJOR)
    for i in range(16):
        assert np.all(A[i, :, i % 8] == 0.0)
        assert d["planted_info"][i] == i % 8 + 1
    assert np.all(np.abs(A[16:]) <= 1.0) and np.all(A[16:] != 0.0)
    _, _, _, info, _ = oracle.getrf_getrs(d["A"], d["B"], ROW_MAJOR, nthreads=NT)
    assert [int(v) for v in info[:16]] == [i % 8 + 1 for i in range(16)]
    assert np.all(info[16:] == 0)


def test_lu_f32_n16_is_standard_normal():
    d = W.make("lu_f32_n16", 4096)
    for a in (d["A"], d["B"]):
        assert a.dtype == np.float32
        assert abs(float(a.mean())) < 0.01 and abs(float(a.std()) - 1.0) < 0.01


def test_chol_f64_n32_planted_minors():
    """About 1% of the systems carry A[k][k] = -1 at a seeded k; the oracle fails them at
    exactly k + 1 (the leading k x k minor is unchanged and positive definite, and the
    k-th Schur value is at most -1), and no other system fails (A = G G^T + 32 I)."""
    d = W.make("chol_f64_n32", 6000)
    planted = d["planted_info"]
    assert 30 <= len(planted) <= 90
    A = from_storage(d["A"], COL_MAJOR)
    for s, code in planted.items():
        assert A[s, code - 1, code - 1] == -1.0
    assert np.array_equal(A, np.swapaxes(A, 1, 2))
    _, _, info = oracle.potrf_potrs(d["A"], d["B"], COL_MAJOR, nthreads=NT)
    want = np.zeros(6000, np.int32)
    for s, code in planted.items():
        want[s] = code
    assert np.array_equal(info, want)


def test_lu_f64_n64_singular_values_and_kappa():
    d = W.make("lu_f64_n64", 40)
    A = from_storage(d["A"], ROW_MAJOR)
    s = np.linalg.svd(A, compute_uv=False)
    kappa = d["kappa"]
    assert np.all((kappa >= 1e2) & (kappa <= 1e8))
    np.testing.assert_allclose(s[:, 0] / s[:, -1], kappa, rtol=1e-6)
    want = 10.0 ** (-np.linspace(0.0, 1.0, 64)[None, :] * np.log10(kappa)[:, None])
    np.testing.assert_allclose(s, want, rtol=1e-6)
    B = d["B"]
    assert np.all(np.abs(B) <= 1.0)


def test_bdsv_systems_are_spd_with_margin():
    """R_i = C_i and L_{i+1} = C_i^T make the assembled matrix symmetric; D_i = M M^T + 10 I
    and |C_i| <= 1/16 entrywise keep its smallest eigenvalue at 9 or more. L_0 and R_last
    are absent (zero); the vector's padding blocks are zero."""
    d = W.make("bdsv_f64_32x8", 6)
    S, x = d["strips"], d["x"]
    bs, nbr = 8, 32
    assert np.all(S[:, 0, :, :bs] == 0) and np.all(S[:, nbr - 1, :, 2 * bs:] == 0)
    assert np.all(np.abs(S[:, :nbr - 1, :, 2 * bs:]) <= 1.0 / 16)
    assert np.all(x[:, :bs] == 0) and np.all(x[:, (nbr + 1) * bs:] == 0)
    dense = W.assemble_bdsv_dense(S)
    assert np.array_equal(dense, np.swapaxes(dense, 1, 2))
    lam = np.linalg.eigvalsh(dense)
    assert np.all(lam[:, 0] >= 9.0)
    _, _, info = oracle.bdsv(S, x, nthreads=NT)
    assert np.all(info == 0)


def test_extra_cholesky_workload_recipe():
    """chol_f64_n256 (the row beyond one CTA): the chol_f64_n32 recipe at n = 256, a
    prefix of the full batch, planted minors at their stated positions, SPD otherwise."""
    d = W.make("chol_f64_n256", 40)
    w = d["workload"]
    assert w.n == 256 and w.nrhs == 1 and w.batch == 2048 and w.layout == W.COL_MAJOR
    A = W.from_storage(d["A"], w.layout)
    assert A.shape == (40, 256, 256) and np.allclose(A, np.swapaxes(A, 1, 2))
    for s, k in d["planted_info"].items():
        assert A[s, k - 1, k - 1] == -1.0
    ok = [s for s in range(40) if s not in d["planted_info"]]
    assert np.all(np.linalg.eigvalsh(A[ok]).min(axis=1) > 200)
    assert np.array_equal(W.make("chol_f64_n256", 20)["A"], d["A"][:20])
