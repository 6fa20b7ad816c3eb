"""The CPU oracle against its pins (see tests/oracle_checks.py)."""
import pytest

import oracle_checks


@pytest.mark.parametrize("check", oracle_checks.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(oracle, check):
    check(oracle)
