"""The oracle's NVFP4 path against brute-force E2M1 / E4M3 searches, hand-derived blocks, a float64
all-experts brute force and invariants (no GPU needed)."""

import pytest

import oracle_nvfp4_pins


@pytest.mark.parametrize("check", oracle_nvfp4_pins.NV_PINS, ids=lambda f: f.__name__)
def test_oracle_nvfp4_pin(check):
    check()
