"""Planted mistakes in the oracle (built as separate copies on the CPU) must
each fail at least one pin, so the pins really constrain the oracle."""
import pytest

import oracle
from _pins import ALL_PINS

# mutant id -> the plausible mistake planted in oracle/attn_oracle.c
MUTANTS = {
    1: "scale dropped from the scores",
    2: "causal mask keeps j < i instead of j <= i",
    3: "softmax not normalised by l",
    4: "off-by-one V row in O = P V",
    5: "LSE missing the row max",
    6: "GQA head mapping h % Hkv instead of h / (H/Hkv)",
    7: "dS missing the D term",
    8: "dS with the wrong sign",
    9: "dK missing the scale",
    10: "e4m3 ties rounded away from zero",
    11: "e4m3 without saturation (NaN code beyond 448)",
    12: "e4m3 subnormal step 2^-8 instead of 2^-9",
    13: "block scale amax / 240 instead of amax / 448",
    14: "V codes not transposed",
    15: "decoding queries aligned top-left instead of bottom-right",
    16: "sliding window one key too wide",
    17: "packed sequences run one row into the next",
    18: "incoherent rotation not normalised by sqrt(d)",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: f"m{m}")
def test_mutant_is_caught(mutant):
    oracle.build(mutant)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mutant=mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches mutant {mutant}: {MUTANTS[mutant]}"
