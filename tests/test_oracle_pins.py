"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle as oracle_mod
from tests import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle):
    pin(oracle)


# Each planted mistake (see ORACLE_PLANT in oracle.c) must be caught by at
# least one pin: a transposed operand, a dropped rank, a wrong sign, an
# off-by-one owner, a skipped canonicalisation, eps outside the square root,
# a chunk count halved by the wrong rule.
@pytest.mark.parametrize("plant", [1, 2, 3, 4, 5, 6, 7])
def test_pins_catch_planted_mistake(plant):
    o = oracle_mod.Oracle(plant=plant)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught planted mistake {plant}"
