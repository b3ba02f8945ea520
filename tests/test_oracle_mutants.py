"""Plant one mistake at a time in the oracle (compiled with -DORACLE_MUTANT=k)
and check that at least one pin catches it. This is how the pins are shown to
be sharp enough: a dropped term, a wrong sign, a wrong index or a transposed
operand anywhere in the oracle fails one of them."""
import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    1: "query head mapped to KV head j % Hkv instead of j / g",
    2: "score scale dropped",
    3: "maximum not subtracted before exp",
    4: "softmax normaliser dropped",
    5: "reads rows 0..n-1 instead of the kept positions",
    6: "last kept token dropped from the value sum",
    7: "value matrix read transposed",
    8: "score sign flipped",
    9: "group pages rounded down",
    10: "group pages sized by the shortest head",
    11: "runs continue on equal instead of consecutive ids",
    12: "gather writes a block to a slot derived from its physical id",
    13: "gather copies one stale block past num_blocks",
    14: "coverage ignores tokens past n",
    15: "budget resolved with max instead of min",
    16: "selection ties broken toward the higher position",
    17: "selection scores with the first query head only",
    18: "recent window one token short",
    19: "reserve run starts one block early",
    20: "released blocks keep their reference",
    21: "alias reads sources after its own writes",
    22: "trim keeps one block past the end",
    23: "reserve fallback takes the highest free blocks",
    24: "trim keeps references to the dropped front blocks",
}


@pytest.mark.parametrize("k", sorted(MUTANTS), ids=[f"m{k}" for k in sorted(MUTANTS)])
def test_mutant_is_caught(k):
    orc = oracle.load_mutant(k)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"mutant {k} ({MUTANTS[k]}) passed every pin"
