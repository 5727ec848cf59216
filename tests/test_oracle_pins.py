"""The float64 oracle against brute force, closed forms and invariants (CPU)."""
import pytest

import oracle_pins
from oracle import latentmoe_ref as ref


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(ref)
