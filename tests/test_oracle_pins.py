"""The CPU oracle against its pins (hand-built words, closed forms, brute force)."""
import pytest

import pins
from oracle import oracle


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)
