"""Each planted mistake in the oracle must fail at least one pin.

The oracle's C source carries compile-time mutants (high nibble first, bias dropped,
sigmoid sign flipped, no renormalisation, wrong scale group, gate and up swapped,
operand rows shifted, shared expert dropped).  Each is compiled here on the CPU and
the pins of test_oracle_pins are run against it: a pin set that let one of them pass
would not pin the oracle.
"""
import pytest

from oracle import Oracle

from test_oracle_pins import ALL_CHECKS

MUTANTS = {
    1: "high nibble first",
    2: "bias term dropped",
    3: "shared-gate sigmoid sign flipped",
    4: "no renormalisation of the top-k",
    5: "wrong scale/bias group index",
    6: "gate and up swapped in SwiGLU",
    7: "matrix rows shifted (transposed operand)",
    8: "shared expert dropped",
    9: "RMSNorm epsilon dropped",
    10: "residual adds the normalised input",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[MUTANTS[m] for m in sorted(MUTANTS)])
def test_mutant_is_caught(mutant):
    o = Oracle(mutant)
    assert o.lib.oracle_mutant() == mutant
    caught = []
    for check in ALL_CHECKS:
        try:
            check(o)
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin catches mutant {mutant} ({MUTANTS[mutant]})"
