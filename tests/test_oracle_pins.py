"""The oracle against its pins (closed forms, a library routine, brute force, invariants)."""
import pytest

import oracle as O
import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(O.load())
