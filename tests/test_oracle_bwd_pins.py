"""The backward oracle against autograd, a closed form and invariants (no GPU needed)."""

import pytest

import oracle_bwd_pins


@pytest.mark.parametrize("check", oracle_bwd_pins.BWD_PINS, ids=lambda f: f.__name__)
def test_oracle_bwd_pin(check):
    check()
