"""Each planted mistake in the oracle (ORACLE_MUTANT=n) must trip a pin.

The mistakes are plausible slips: a dropped scale, a flipped exponent sign,
a value row paired with the wrong key, ties sent the wrong way, the lowest
scores kept, one head of a group scored, padding read as a position, a stale
selection reused, a missing normaliser, one position short, a shifted
feature index."""
import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = [1, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_mutant_is_caught(mutant):
    orc = oracle.get(mutant)
    assert orc.mutant_id() == mutant
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
