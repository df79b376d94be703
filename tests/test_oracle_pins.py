"""The CPU oracle against its pins (closed forms, hand-worked examples,
exact-rational brute force, invariants, independent library routines)."""
import pytest

import pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    check(orc)
