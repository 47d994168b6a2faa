"""The CPU oracle against its pins (no GPU needed), plus the mutation check: every
deliberately broken build of the oracle must fail at least one pin."""
import pytest

import oracle
from oracle_pins import PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.load(0)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("mutant", sorted(oracle.MUTANTS), ids=lambda m: f"m{m}")
def test_mutant_is_caught(mutant):
    mut = oracle.load(mutant)
    assert mut.mutant == mutant
    failed = []
    for pin in PINS:
        try:
            pin(mut)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({oracle.MUTANTS[mutant]}) passed every pin"
