"""The oracle against its pins (brute force, closed forms, invariants, special
cases); see oracle_pins.py for what each pin checks."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)
