"""Pins of the fp64 oracle (CPU only): every check in _pins.py must hold."""
import pytest

import _pins


@pytest.mark.parametrize("check", _pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, check):
    check(orc)
