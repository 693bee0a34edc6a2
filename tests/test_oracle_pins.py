"""The CPU oracle against closed forms, brute force, finite differences, torch
float64, the vocabulary-split combine and exhaustive rounding (CPU only)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)
