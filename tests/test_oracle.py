"""The CPU oracle against its pins (no GPU): hand-derived cases, closed forms,
invariants and an independent complex-exponential evaluation of the rotation.
See ``oracle_pins.py`` for what each pin fixes."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from oracle_pins import ALL_PINS  # noqa: E402


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)
