"""The oracle against its pins (CPU only)."""
import pytest

import oracle
from tests import oracle_pins

CHECKS = oracle_pins.all_checks()


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_oracle_pin(check):
    check(oracle)
