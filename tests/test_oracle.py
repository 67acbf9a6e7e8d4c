"""The oracle against its pins (CPU only): golden hand rows, exact rational
results, closed forms, invariants and float64 brute force."""
import pytest

import oracle
from oracle_pins import PINS


@pytest.fixture(scope="module")
def O():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(O, pin):
    pin(O)


def test_oracle_rejects_bad_arguments(O):
    import numpy as np
    x = np.zeros((2, 4), np.uint16)
    with pytest.raises(ValueError):
        O.forward([x], np.zeros((2, 5), np.uint16), np.zeros(4, np.uint16), 1e-6)
    with pytest.raises(ValueError):
        O.forward([x], x, np.zeros(3, np.uint16), 1e-6)


def test_oracle_empty_rows(O):
    import numpy as np
    x = np.zeros((0, 8), np.uint16)
    red, ro, nrm = O.forward([x, x], x, np.zeros(8, np.uint16), 1e-6)
    assert red.shape == ro.shape == nrm.shape == (0, 8)
