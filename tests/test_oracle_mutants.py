"""Pin strength: each planted mistake in the oracle (a dropped term, a wrong
sign, a shifted causal index, eps in the wrong place, swapped operands) must
make at least one pin fail.  The mistakes are compiled into separate copies
of the C oracle on the CPU; the real oracle is untouched."""
import pytest

import oracle
import oracle_pins

MUTANTS = {
    1: "log sigma2 term dropped",
    2: "distance divided by sigma, not sigma^2",
    3: "exclusive causal prefix",
    4: "eps in the numerator",
    5: "query/key responsibilities swapped",
    6: "prior with the wrong sign",
    9: "decode step reads before its key enters the memory",
    10: "usage counts hard assignments",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_pins_catch_planted_mistake(mutant):
    caught = []
    with oracle.use_mutant(mutant):
        for pin in oracle_pins.ALL_PINS:
            try:
                pin()
            except AssertionError:
                caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {mutant} ({MUTANTS[mutant]})"
