"""Each build of the oracle with one planted bug must fail at least one pin."""
import pytest

from tests import oracle_pins as P


@pytest.mark.parametrize("mutant", sorted(P.MUTANTS), ids=lambda m: f"m{m}-{P.MUTANTS[m].replace(' ', '_')}")
def test_some_pin_rejects_mutant(mutant):
    failures = []
    for pin in P.ALL_PINS:
        try:
            pin(mutant=mutant)
        except AssertionError:
            failures.append(pin.__name__)
    assert failures, f"no pin caught mutant {mutant}: {P.MUTANTS[mutant]}"
