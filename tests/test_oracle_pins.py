"""The CPU oracle against library routines, closed forms and invariances."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(olib, pin):
    pin(olib)
