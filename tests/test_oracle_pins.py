"""The oracle against its pins (closed forms, invariants, library rounding, brute force)."""

import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.kda_oracle)
