"""The oracle against its pins (brute force, library special cases, closed
forms, hand-worked tables, invariants). CPU only."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_oracle_rejects_bad_layout_input(orc):
    import numpy as np

    from oracle import OracleError

    with pytest.raises(OracleError):
        orc.layout(np.array([[1, 1]], np.int32), 4, 2)  # same expert twice in one token
    with pytest.raises(OracleError):
        orc.layout(np.array([[0, 4]], np.int32), 4, 2)  # expert out of range
    with pytest.raises(OracleError):
        orc.layout(np.array([[0, 1]], np.int32), 6, 4)  # E % R != 0
