"""The oracle against its pins (CPU only). See tests/pins.py for what each pin
compares the oracle with."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()
