"""The fp64 oracle against its pins (special cases, closed forms, invariants)."""
import pytest

import oracle
from pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.default())


def test_threads_do_not_change_result():
    """Column blocking over threads is exact: 1 thread and many agree bit for bit."""
    import numpy as np
    from pins import _rand_case
    rng = np.random.default_rng(5)
    q, k, v, la, b = _rand_case(rng, 50, 3, 16, 32)
    s0 = rng.standard_normal((1, 3, 16, 32))
    o1, s1 = oracle.prefill(q, k, v, la, b, None, s0, threads=1)
    o2, s2 = oracle.prefill(q, k, v, la, b, None, s0, threads=7)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)
