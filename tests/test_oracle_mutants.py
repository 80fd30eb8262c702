"""Each planted mistake in the oracle (ORACLE_MUTANT builds of the same C file)
must fail at least one pin — evidence that the pins would catch a dropped term,
a wrong sign, index or tie-break.  CPU only."""
import pytest

import oracle
import pins

MUTANTS = {
    1: "projection reads W transposed",
    2: "binarisation threshold >= 0",
    3: "only the first query head of a group is scored",
    4: "ties go to the highest slot",
    5: "evicts the most similar slot",
    6: "attention scale 1/sqrt(D) dropped",
    7: "value rows read with a transposed index",
    8: "the new token's value is not written",
    9: "score memory weighs the new distance instead of the old score",
    10: "the written slot keeps the evicted token's score",
    11: "binarisation threshold with the wrong sign",
    12: "score ties go to the highest slot",
    13: "value rows scaled by max / 128",
    14: "value rows rounded half away from zero",
    15: "a chunk scores by its first slot only",
    16: "staged tokens land in reverse order",
    17: "a chunk scores its slots shifted by one",
    18: "fp8 values: ties rounded away from zero",
    19: "fp8 value rows scaled by max / 256",
    20: "fp8 subnormals decoded with the implicit leading bit",
    21: "median thresholds take the upper median",
    22: "bit j compared with the threshold of bit j + 1",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_mutant_is_caught(mutant, tmp_path_factory):
    o = oracle.load(mutant, build_dir=str(tmp_path_factory.mktemp(f"mut{mutant}")))
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(o)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
