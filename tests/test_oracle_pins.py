"""The fp64 oracle against facts the pages and the mathematics fix (CPU only)."""
import pytest

import oracle
from tests import _pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, lib):
    pin(lib)
