"""The fp64 oracle against values and facts fixed outside it (CPU only)."""
import pytest

from oracle import rmsnorm_oracle
from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(rmsnorm_oracle)
