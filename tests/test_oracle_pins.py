"""The CPU oracle against facts outside itself (see oracle_pins.py)."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def o():
    return oracle.load()


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(o, pin):
    pin(o)


def test_rejects_bad_sizes(o):
    import numpy as np
    with pytest.raises(ValueError):
        o.matmul_q4_0(np.zeros((1, 48), np.float32), np.zeros(18, np.uint8), 1, 48)
    rc = o.lib.oracle_matmul_q4_0(None, None, 1, 1, 33, None, None)
    assert rc == -1
