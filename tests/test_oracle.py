"""The fp64 oracle against facts outside itself (CPU only)."""
import pytest

import oracle.fp64 as O
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(O)
