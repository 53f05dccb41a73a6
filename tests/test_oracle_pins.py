"""The CPU oracle against its pins (hand tables, closed forms, brute force)."""
import pytest

from oracle import moe_oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(moe_oracle)
