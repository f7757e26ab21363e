"""The oracle against its pins (CPU only).  See ``oracle_pins.py`` for what each pins."""
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__[4:])
def test_pin(pin, lib):
    pin(lib)
