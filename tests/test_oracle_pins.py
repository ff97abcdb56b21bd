"""The CPU oracle against its pins (closed forms, library routines, brute force,
invariants).  No GPU needed."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_default):
    pin(oracle_default)
