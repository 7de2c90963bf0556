"""The oracle against brute force, closed forms, library routines and invariants."""
import pytest

import oracle_pins

PINS = sorted(n for n in dir(oracle_pins) if n.startswith("pin_"))


@pytest.mark.parametrize("name", PINS)
def test_pin(name):
    getattr(oracle_pins, name)()
