"""The oracle against its pins (values fixed by the pages and by mathematics)."""
import pytest

import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(ora, pin):
    pin(ora)
