"""The CPU oracle against checks that do not come from the oracle itself.

See tests/pins.py for what each pin computes and why it is independent.
"""

import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)
