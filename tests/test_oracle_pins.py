"""The fp64 oracle against its pins (CPU only).

Every pin is described in ``oracle_pins.py``; each compares the oracle with a
hand-derived worked example, a closed form, an invariant or a one-hot special
case of the mHC equations (page "mHC 算法分析 & cutile 高效实现", §2).
"""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()
