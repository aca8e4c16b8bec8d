"""The committed oracle against every pin (printed values, closed forms, invariants,
library special cases, brute force).  CPU only."""
import pytest

from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)
