"""The fp64 oracle against its pins (CPU only)."""
import pytest

from oracle import oracle as orc
from tests.pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(orc._default)
