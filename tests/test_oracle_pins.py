"""The oracle against its pins (CPU only); see tests/pins.py for what each rests on."""
import pytest

import oracle
from tests import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.default())


def test_oracle_thread_count_does_not_change_results():
    """The batch loop only hands whole systems to worker threads."""
    import numpy as np
    from gen import workloads as W
    d = W.make("lu_f32_n16", batch=500)
    a = oracle.getrf_getrs(d["A"], d["B"], oracle.ROW_MAJOR, nthreads=1)
    b = oracle.getrf_getrs(d["A"], d["B"], oracle.ROW_MAJOR, nthreads=7)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    d = W.make("chol_f64_n32", batch=300)
    a = oracle.potrf_potrs(d["A"], d["B"], oracle.COL_MAJOR, nthreads=1)
    b = oracle.potrf_potrs(d["A"], d["B"], oracle.COL_MAJOR, nthreads=5)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    d = W.make("bdsv_f64_32x8", batch=40)
    a = oracle.bdsv(d["strips"], d["x"], nthreads=1)
    b = oracle.bdsv(d["strips"], d["x"], nthreads=3)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
