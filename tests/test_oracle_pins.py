"""The oracle against its pins (CPU only), and the pins against planted mistakes."""
import pytest

import oracle as oracle_pkg
from oracle_pins import ALL_PINS, MUTANTS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(oracle, pin):
    pin(oracle)


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[MUTANTS[m] for m in sorted(MUTANTS)])
def test_planted_mistake_is_caught(mutant):
    orc = oracle_pkg.load(mutant)
    assert orc.mutant == mutant
    tripped = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            tripped.append(pin.__name__)
    assert tripped, f"planted mistake '{MUTANTS[mutant]}' passed every pin"
