"""The fp64 oracle against its pins (closed forms, invariants, brute force,
textbook library routines) -- see ``oracle_pins.py`` for what each checks."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()
