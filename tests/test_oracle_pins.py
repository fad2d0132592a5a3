"""The fp64 oracle against facts fixed outside itself (CPU only).

See tests/oracle_pins.py for what each check pins and where it comes from.
"""

import pytest

import oracle
from oracle_pins import ALL_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle)
