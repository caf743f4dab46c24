"""The CPU oracle against facts that do not come from it (see ``_pins.py``)."""
import pytest

import oracle
import _pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", _pins.PINS, ids=lambda p: p.__name__)
def test_pin(pin, lib):
    pin(lib)
