"""The CPU oracle against its pins (no GPU)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=[p.__name__ for p in pins.ALL_PINS])
def test_pin(pin, oracle_lib):
    pin()


def test_oracle_rejects_bad_values(oracle_lib):
    import numpy as np
    O = oracle_lib
    with pytest.raises(O.OracleError):
        O.pack_i2s(np.full((1, 128), 2, np.int8), 1.0)
    with pytest.raises(O.OracleError):
        O.pack_i2s(np.zeros((1, 100), np.int8), 1.0)
    bad = np.full(32 + 4, 0xFF, np.uint8)          # code 0b11 is never produced by i2_s
    with pytest.raises(O.OracleError):
        O.unpack_i2s(bad, 1, 128)
    badt = np.zeros(66, np.uint8)
    badt[0] = 0b10                                  # TQ2_0 code 0b10 is never produced
    with pytest.raises(O.OracleError):
        O.unpack_tq2_0(badt, 1, 256)
    with pytest.raises(O.OracleError):
        O.pack_w1(np.full((1, 32), 3, np.int8))
