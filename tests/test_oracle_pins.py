"""The CPU oracle against facts other than itself (no GPU needed)."""

import pytest

from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(oracle, pin):
    pin(oracle)
