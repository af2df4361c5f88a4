"""The fp64 oracle against facts that do not come from the oracle (CPU only)."""
import pytest

import oracle
from oracle_checks import ALL_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle)
