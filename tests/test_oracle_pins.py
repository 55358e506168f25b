"""The CPU oracle against its pins (no GPU).

Every pin is defined in ``oracle_pins.py``; see there for what each one ties
the oracle to.
"""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)
