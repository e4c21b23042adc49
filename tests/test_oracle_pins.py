"""The CPU oracle against its pins (no GPU needed)."""

import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    oracle.load()
    pin(oracle.LIB)


def test_oracle_rejects_bad_arguments():
    import numpy as np
    orc = oracle.Oracle(4, 2, 1)  # k_heavy + k_local != budget
    st = orc.new_state(1, 4, np.float32)
    x = np.zeros((1, 3, 4), dtype=np.float32)
    with pytest.raises(ValueError):
        orc.prefill_select(x, x, x, st)
    orc = oracle.Oracle(4, 2, 2)
    st = orc.new_state(1, 4, np.float32)
    z = np.zeros((1, 4), dtype=np.float32)
    with pytest.raises(ValueError):  # slot map does not hold min(t, budget) valid slots
        orc.decode_step(3, z, z, z, st)
