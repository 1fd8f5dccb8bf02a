"""The CPU oracle against facts that do not come from the oracle itself."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_mod, pin):
    pin()
