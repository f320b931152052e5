"""The fp64 oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

from _pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(mutant=0)
