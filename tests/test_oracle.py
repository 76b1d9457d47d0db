"""CPU tests: the float64 oracle against its pins (no GPU, no library code)."""

import pytest

import oracle
import oracle.fp8
from tests import oracle_pins, oracle_pins_fp8


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle)


@pytest.mark.parametrize("pin", oracle_pins_fp8.FP8_PINS, ids=lambda f: f.__name__)
def test_oracle_fp8_pin(pin):
    pin(oracle.fp8)
