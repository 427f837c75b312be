"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle
from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(oracle.attention)


from tests.oracle_pins_fp8 import FP8_PINS  # noqa: E402
import oracle.fp8  # noqa: E402


@pytest.mark.parametrize("pin", FP8_PINS, ids=[p.__name__ for p in FP8_PINS])
def test_fp8_pin(pin):
    pin(oracle.fp8)
