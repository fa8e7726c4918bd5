"""The oracle against its pins (closed forms, invariants, brute force, page values)."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.get(0)


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_oracle_is_the_unmutated_build(orc):
    assert orc.mutant_id() == 0
