"""The CPU oracle against facts fixed outside itself (no GPU needed)."""
import pytest

from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(orc, pin):
    pin(orc)


def test_oracle_rejects_bad_arguments(orc):
    import numpy as np
    A = np.zeros((3, 4), np.float32)
    B = np.zeros((5, 2), np.float32)
    with pytest.raises(ValueError):
        orc.sgemm_f64(0, 0, 1.0, A, B)          # K mismatch
    with pytest.raises(ValueError):
        orc.sgemm_f64(2, 0, 1.0, A, B)          # bad op
