"""Planted mistakes in the oracle must each fail at least one pin (no GPU).

Each mutant is the oracle compiled with -DKDO_MUTANT=<n>; the mistakes are
listed in oracle/kdt_oracle.c."""
import pytest

import oracle
import _pins

MUTANTS = {
    1: "split rank off by one",
    2: "super key not cyclic",
    3: "index tiebreak reversed",
    4: "widest-dimension ties go to the highest dimension",
    5: "left and right subtrees swapped",
    6: "left child domain clipped on the wrong side",
    7: "round-robin phase shifted by one level",
    8: "balanced tree: upper median instead of lower",
    9: "balanced tree: subtrees swapped",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_mutant_is_caught(mutant):
    o = oracle.Oracle(mutant)
    failed = []
    for pin in _pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
        except oracle.OracleError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
