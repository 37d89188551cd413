"""Each planted mistake in the oracle (a dropped term, a wrong sign, a swapped
operand, a wrong index or tie rule, a wrong rounding) must fail at least one
pin.  The mistakes are compiled into copies of the oracle on the CPU
(ORACLE_MUTANT=n); the oracle used everywhere else is built with n = 0."""
import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    1: "up projection dropped",
    2: "wrong sign inside SiLU",
    3: "gate and up swapped",
    4: "top-k ties to the higher id",
    5: "shared expert dropped",
    6: "weights not renormalised",
    7: "group order reversed",
    8: "inclusive instead of exclusive scan",
    9: "combine uses the next slot's weight",
    10: "router bias subtracted",
    11: "bf16 rounding truncates",
    12: "chosen set listed in descending id",
    13: "E4M3 encoding truncates",
    14: "activation full-scale value 440 instead of 448",
    15: "FP8 activation scale dropped from the gate/up sums",
    16: "E2M1 rounding ties away from zero",
    17: "NVFP4 row scale without the block range 6",
    18: "NVFP4 block scales indexed as 32-wide blocks",
    19: "NVFP4 down-projection tensor scale dropped",
    20: "NVFP4 linear layer drops the row scale",
    21: "E4M3 linear layer drops the weight scale",
}


@pytest.mark.parametrize("n", sorted(MUTANTS), ids=lambda n: f"m{n}")
def test_mutant_is_caught(n, tmp_path):
    lib = oracle.build(mutant=n, out_dir=tmp_path)
    o = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
        except Exception:            # e.g. an index error from a broken offset table
            caught.append(pin.__name__ + " (error)")
    assert caught, f"no pin caught mutant {n}: {MUTANTS[n]}"
