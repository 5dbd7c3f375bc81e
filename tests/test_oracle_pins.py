"""The CPU oracle against brute force, closed forms and invariants (no GPU needed)."""

import pytest

import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()
