"""The CPU oracle against facts that do not come from the oracle (CPU only)."""
import pytest

from tests.oracle_pins import CHECKS


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_oracle_pin(orc, check):
    check(orc)
