"""Planted mistakes in the oracle (built with -DHWREF_MUTANT=n, on the CPU):
each must fail at least one pin, which shows that the pins can see it."""
import pytest

import oracle
from tests import oracle_pins as P

MUTANTS = {
    1: "rotation in the wrong direction",
    2: "wrong frequency exponent",
    3: "adjacent pairing instead of rotate_half",
    4: "query rotated by i_q + offset",
    5: "lse without the max term",
    6: "strided GQA head mapping",
    7: "commit places tokens in reverse order",
    8: "commit rotates by -delta",
    9: "a limited entry leaves out its last visible token",
    10: "E4M3 exponent bias off by one",
    11: "E4M3 keys scaled by another head's scale",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_mutant_is_caught(mutant):
    o = oracle.get(mutant)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
