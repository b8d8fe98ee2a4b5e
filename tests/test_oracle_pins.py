"""The CPU oracle against facts fixed by the format definitions (see pins.py)."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def ora():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(ora, pin):
    pin(ora)
