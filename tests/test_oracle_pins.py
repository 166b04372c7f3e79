"""The CPU oracle against its pins (see oracle_pins.py); no GPU needed."""
import pytest

from .oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)
