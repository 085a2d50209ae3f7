"""The oracle against its pins (CPU only).

See tests/oracle_pins.py for what each pin checks and why it is independent of
the oracle's own code.
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
