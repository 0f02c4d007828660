"""The fp64 oracle against its pins (no GPU).

Every function in ``tests/oracle_pins.py`` checks the oracle against a value a
page prints, a closed form, an invariant, an independent library routine or a
different algorithm for the same quantity.
"""
import numpy as np
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_pin(pin, lib):
    pin(lib)


def test_naive_softmax_overflows():
    """Why the oracle shifts by the maximum: the unshifted formula of the
    stable-softmax lesson (section 一) overflows to inf/inf = NaN on 1000, 999, 998,
    even in double."""
    x = np.array([1000.0, 999.0, 998.0])
    with np.errstate(over="ignore", invalid="ignore"):
        naive = np.exp(x) / np.exp(x).sum()
    assert np.all(np.isnan(naive))
    y = oracle.softmax_rows([x])[0]
    assert np.all(np.isfinite(y))


def test_oracle_threads():
    assert oracle.num_threads() >= 1


def test_empty_inputs(lib):
    y = oracle.softmax_rows(np.zeros((0, 5), np.float32), lib=lib)
    assert y.shape == (0, 5)
    Q = np.zeros((0, 2, 4), np.float32)
    O, lse = oracle.attention_packed(Q, Q, Q, [0], 0.5, True, lib=lib)
    assert O.shape == (0, 2, 4) and lse.shape == (2, 0)
