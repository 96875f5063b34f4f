"""The oracle against its pins (CPU only)."""
import pytest

import oracle
from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(oracle.default())


def test_cu_seqlens_validation():
    import numpy as np

    q = np.zeros((4, 1, 2))
    with pytest.raises(ValueError):
        oracle.recurrence(q, q, q, q, np.zeros((4, 1)), cu_seqlens=[0, 3, 2, 4])
    with pytest.raises(ValueError):
        oracle.recurrence(q, q, q, q, np.zeros((4, 1)), cu_seqlens=[0, 3])
