"""The float64 oracle against the pages' worked examples, closed forms,
invariants, a library routine and finite differences (no GPU)."""
import pytest

import oracle.ref as ref
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(ref)
