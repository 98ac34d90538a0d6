"""The oracle against its pins: the pages' worked examples and test catalog,
closed forms, invariants, brute force and library special cases (CPU only)."""
import pytest

import pins


@pytest.mark.parametrize("name", sorted(pins.PINS))
def test_pin(orc, name):
    pins.PINS[name](orc)
