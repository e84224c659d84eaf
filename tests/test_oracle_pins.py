"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import oracle.moe_oracle as oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle)
