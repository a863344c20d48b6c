"""The oracle against its pins (CPU only)."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(__file__))

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle)
