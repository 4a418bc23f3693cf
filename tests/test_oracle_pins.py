"""The CPU oracle against its pins (hand-worked goldens, exact rational
re-derivation, invariants, special cases, brute-force placement)."""
import pytest

import _pins


@pytest.mark.parametrize("pin", _pins.PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)
