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


def test_oracle_rejects_bad_kept_sets(orc):
    import numpy as np
    q = np.zeros((1, 4))
    k = np.zeros((5, 4))
    with pytest.raises(ValueError):
        orc.attn_head(q, k, k, np.array([3, 1], np.int32), 1.0)   # not ascending
    with pytest.raises(ValueError):
        orc.attn_head(q, k, k, np.array([5], np.int32), 1.0)      # out of range
    with pytest.raises(ValueError):
        orc.resolve_budget(np.array([[0]], np.int32), np.array([3], np.int32))
