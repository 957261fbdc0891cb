"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

from oracle import moe_oracle
from tests.oracle_pins import ALL_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(moe_oracle)
