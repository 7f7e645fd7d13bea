"""The CPU oracle against its pins (hand-worked fixtures, brute force, closed forms, invariants)."""
import pytest

import oracle.moe as oracle_moe
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(oracle_moe)
