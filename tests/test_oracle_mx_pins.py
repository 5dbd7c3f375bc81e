"""The oracle's MXFP8 path against brute force, torch's float8 cast, hand-derived blocks and
invariants (no GPU needed)."""

import pytest

import oracle_mx_pins


@pytest.mark.parametrize("check", oracle_mx_pins.MX_PINS, ids=lambda f: f.__name__)
def test_oracle_mx_pin(check):
    check()
