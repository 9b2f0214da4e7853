"""The oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

from oracle_pins import ALL_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check, oracle_lib):
    check(oracle_lib)
