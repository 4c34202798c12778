"""The fp64 oracle against its pins (closed forms, special cases, a
hand-derived worked example); CPU only."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load())


def test_rejects_bad_arguments():
    import numpy as np
    with pytest.raises(ValueError):
        oracle.scan_fwd(np.zeros((1, 2, 3)), np.zeros((1, 2, 4)), np.zeros((3, 2)),
                        np.zeros((1, 2, 2)), np.zeros((1, 2, 2)))
