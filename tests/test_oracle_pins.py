"""The oracle against facts that do not come from the oracle itself."""
import pytest

import oracle_pins
from oracle import moe_oracle


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(moe_oracle)
