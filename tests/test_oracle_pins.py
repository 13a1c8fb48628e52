"""The oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

from oracle_pins import ALL_PINS
from oracle_pins_powersgd import POWERSGD_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("pin", POWERSGD_PINS, ids=[p.__name__ for p in POWERSGD_PINS])
def test_powersgd_pin(orc, pin):
    from oracle import powersgd

    pin(orc, powersgd)
