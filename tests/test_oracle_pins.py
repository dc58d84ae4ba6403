"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle
from oracle_pins import ALL_CHECKS


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("check", ALL_CHECKS, ids=[c.__name__ for c in ALL_CHECKS])
def test_oracle_pin(check, lib):
    check(lib)
