"""The CPU oracle against facts fixed independently of it (see oracle_pins)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_rejects_bad_arguments(orc):
    import numpy as np
    W = np.zeros((2, 48), dtype=np.uint16)
    with pytest.raises(ValueError):
        orc.prune_pack(W, 2, 4)          # cols not a multiple of 32
    W = np.zeros((2, 64), dtype=np.uint16)
    for N, M in [(1, 4), (3, 4), (2, 8), (8, 32), (32, 64), (0, 0)]:
        with pytest.raises(ValueError):
            orc.prune_pack(W, N, M)
    values = np.zeros((1, 32), dtype=np.uint16)
    masks = np.array([[0xFFFF, 0x1]], dtype=np.uint32)  # second word popcount 1
    with pytest.raises(ValueError):
        orc.unpack(values, masks, 64)
