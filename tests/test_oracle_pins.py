"""The CPU oracle against values and properties fixed outside itself (CPU only)."""
import pytest

import oracle_pins as pins
from oracle import Oracle


@pytest.fixture(scope="module")
def o():
    return Oracle()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(o, pin):
    pin(o)


def test_nonfinite_logits_rejected(o):
    import numpy as np
    from oracle import OracleError
    logits = np.array([[0.0, np.nan, 1.0]], np.float32)
    with pytest.raises(OracleError):
        o.route(logits, 2, True)


def test_page_outside_pool_rejected(o):
    import numpy as np
    from oracle import OracleError
    pool = np.zeros(4 * 64, np.uint8)
    with pytest.raises(OracleError):
        o.page_to_matrix(pool, 64, 4, 4, 4)
    with pytest.raises(OracleError):
        o.page_to_matrix(pool, 64, 0, 8, 8)  # 128 bytes do not fit a 64-byte page
