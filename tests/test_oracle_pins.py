"""The CPU oracle against its pins (hand-worked fixtures, closed forms, special
cases, brute force).  CPU only."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def o():
    return oracle.load()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(o, check):
    check(o)


def test_simhash_law(o):
    pins.check_simhash_law(o)
