"""The CPU oracle against its pins, and every planted mistake against them.

CPU only.  See tests/oracle_pins.py for what each pin checks and why it is
independent of the oracle's own code.
"""
import tempfile

import pytest

import oracle
from tests import oracle_pins as P


@pytest.mark.parametrize("pin", P.PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


# Planted mistakes (ORC_MUTANT in q4_oracle.c):
#  1 swapped nibble halves, 2 dropped -8 offset, 3 ties-to-even rounding,
#  4 inverse scale from the fp16 d, 5 activation scale dropped,
#  6 wrong activation block index, 7 signed instead of absolute max,
#  8 truncating fp16 encode, 9 argmax ties to the highest index,
#  10 transposed output, 11 top-2 second ties to the highest index,
#  12 verify rule comparing a draft with its own prediction,
#  13 Q8_0 weights read as unsigned, 14 SiLU with exp(+g),
#  15 Q4_0 encoder scale from the magnitude, 16 Q4_0 codes rounded down,
#  17 Q8_0 weights read as unsigned when requantised to Q4_0,
#  18 the epilogue's residual of token 0 used for every token,
#  19 gs64 nibbles read as GGML-style pairs, 20 the per-vector activation
#  scale from the first block's maximum only.
MUTANTS = list(range(1, 21))


@pytest.fixture(scope="module")
def mutdir():
    with tempfile.TemporaryDirectory(prefix="orc_mut_") as d:
        yield d


@pytest.mark.parametrize("m", MUTANTS)
def test_pins_reject_mutant(mutdir, m):
    o = oracle.Oracle(oracle.build_mutant(m, mutdir))
    assert o.mutant() == m
    failed = []
    for pin in P.PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {m} passed every pin"
