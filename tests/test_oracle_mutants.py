"""Plant mistakes in the oracle (on the CPU) and check that the pins catch each one.

Each mutant is cpr_oracle.c compiled with ORACLE_MUTANT=n: a flipped sign, a dropped
decay, a dropped beta, the output taken before the update, a transposed state, a
wrongly signed exponent, boundary states one token late, a wrong decay in the chunk
update, a dropped decay vector, a wrong final state for a partial chunk.
"""
import pytest

import _pins
import oracle

MUTANTS = list(range(1, 11))


@pytest.mark.parametrize("mutant", MUTANTS)
def test_pins_catch_mutant(mutant):
    oracle.build(mutant)
    failed = []
    for pin in _pins.ALL_PINS:
        try:
            ok, detail = pin(mutant=mutant)
        except Exception as e:  # a crash also counts as caught
            ok, detail = False, repr(e)
        if not ok:
            failed.append(f"{pin.__name__}: {detail}")
    assert failed, f"no pin caught oracle mutant {mutant}"
