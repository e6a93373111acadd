"""The fp64 oracle against facts fixed outside itself (CPU only)."""
import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS,
                         ids=[c.__name__ for c in oracle_pins.ALL_CHECKS])
def test_oracle_pin(check):
    check(oracle.default())
