"""The oracle against its pins (CPU only)."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(orc, pin):
    pin(orc)


def test_fwd_no_residual_has_no_new_residual(orc):
    import numpy as np
    out, new_res = orc.fwd(np.ones((2, 3)), np.ones(3), 1e-5)
    assert new_res is None and out.shape == (2, 3)


def test_scalars_are_float32(orc):
    """eps and weight_bias reach the oracle as the float32 values the CUDA
    library sees."""
    import numpy as np
    assert orc.scalar(1e-5) == float(np.float32(1e-5))
    assert orc.scalar(0.1) != 0.1
