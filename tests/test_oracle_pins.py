"""The oracle against facts that do not come from the oracle itself."""
import pytest

import head_pins
import oracle_pins
from oracle import head_oracle, moe_oracle


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(moe_oracle)


@pytest.mark.parametrize("pin", head_pins.ALL_HEAD_PINS, ids=lambda p: p.__name__)
def test_head_pin(pin):
    pin(head_oracle)
