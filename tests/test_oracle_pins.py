"""The CPU oracle against its pins (no GPU): hand-worked values, library
routines, invariants, closed forms and error bounds.  Then the same pins run
against oracle builds with one planted mistake each, and must reject all."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_lib, check):
    check(oracle_lib)


MUTANTS = {
    1: "channel size rounded down instead of up",
    2: "block offset uses the source rank's own prefix (off by one)",
    3: "combine sums in descending rank order",
    4: "node-level receive prefix reads the transposed peer",
    5: "per-expert count rounded down to the alignment",
    6: "received top-k ids left global",
    7: "a token counted once per slot instead of once per rank",
    8: "bf16 conversion truncates instead of rounding",
    9: "LL combine rounds the product before adding (no fused multiply-add)",
    10: "LL layout visits a token's slots in descending order",
    11: "combine weights summed in descending rank order",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: f"mutant{m}")
def test_pins_reject_planted_mistake(mutant):
    o = oracle.load(mutant=mutant)
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(o)
        except (AssertionError, ValueError, IndexError):
            caught.append(check.__name__)
    assert caught, f"no pin caught mutant {mutant}: {MUTANTS[mutant]}"
