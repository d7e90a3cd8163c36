"""Each planted mistake in the oracle is caught by at least one pin (CPU only).

The mistakes are compiled into separate builds of the oracle's C source
(ORACLE_MUTANT=n): swapped nibbles, ties-to-even rounding, wrong sign of d,
last-index tie break, dropped -8 offset, transposed x index, division by the
stored fp16 d, truncating fp16 encoder, dropped last k term, the scale's
two bytes swapped, codes clamped at 14.
"""
import pytest

import oracle
import pins

MUTANTS = {1: "nibbles swapped", 2: "round ties to even", 3: "sign of d flipped",
           4: "last index wins max tie", 5: "offset 8 dropped", 6: "x index transposed",
           7: "divide by stored fp16 d", 8: "fp16 encoder truncates", 9: "last k term dropped",
           10: "scale bytes swapped", 11: "codes clamped at 14"}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_mutant_is_caught(mutant, tmp_path):
    o = oracle.Oracle(mutant=mutant, out_dir=str(tmp_path))
    assert o.lib.oracle_mutant() == mutant
    failed = []
    for pin in pins.FAST_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
