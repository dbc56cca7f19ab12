"""Planted mistakes in the oracle must each trip at least one pin.

Each mutant is the oracle's C source compiled with -DORACLE_MUTANT=k, which
breaks exactly one step: 1 flips the adjoint's exponent sign, 2 drops the
kz*z term, 3 transposes Dr and Di, 4 flips a sign of the complex multiply,
5 reads the wrong coordinate, 6 uses pi instead of 2 pi, 7 skips the first
sample, 8 gives the forward operator the adjoint's sign.
"""
import pytest

import oracle
from tests.oracle_pins import ALL_PINS

MUTANTS = [1, 2, 3, 4, 5, 6, 7, 8]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_mutant_is_caught(mutant):
    orc = oracle.Oracle(mutant)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
