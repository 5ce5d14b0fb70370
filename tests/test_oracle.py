"""The fp64 oracle against closed forms, invariants, brute force and library routines."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, lib):
    pin(lib)


def test_threads_do_not_change_results(lib):
    import numpy as np

    g = np.random.default_rng(0)
    q, k, v = (g.standard_normal((4, 33, 8)) for _ in range(3))
    oracle.set_threads(1)
    o1, l1 = oracle.attention(q, k, v, True, 0.5)
    oracle.set_threads(4)
    o4, l4 = oracle.attention(q, k, v, True, 0.5)
    oracle.set_threads(1)
    assert (o1 == o4).all() and (l1 == l4).all()
