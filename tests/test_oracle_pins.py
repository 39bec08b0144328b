"""The CPU oracle against what the pages' formulas and mathematics fix (no GPU)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)
