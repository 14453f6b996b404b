"""The CPU oracle against its pins (closed forms, hand-derived cases, numpy)."""
import pytest

import oracle
from oracle_pins import ALL_CHECKS


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    check(orc)
