"""The oracle against its pins (CPU only): library routines, textbook rounding,
closed forms, brute force and invariants -- see pins.py for each fact."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("name", sorted(pins.ALL_CHECKS))
def test_oracle_pin(name):
    pins.ALL_CHECKS[name](oracle.default())
