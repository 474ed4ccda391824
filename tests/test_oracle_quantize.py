"""The oracle's quantiser against its pins, and planted mistakes in a copy of
it (on the CPU), each of which some pin must catch."""
import os
import shutil

import pytest

import oracle
from quant_pins import QUANT_PINS


@pytest.mark.parametrize("pin", QUANT_PINS, ids=lambda p: p.__name__)
def test_quantizer_pin(pin, orc):
    pin(orc)


QUANT_MUTATIONS = {
    "zero_point_7": [("float t = rintf(w[j] / d) + 8.0f;", "float t = rintf(w[j] / d) + 7.0f;")],
    "truncate_not_round": [("float t = rintf(w[j] / d) + 8.0f;", "float t = truncf(w[j] / d) + 8.0f;")],
    "positive_scale_from_magnitude": [("oracle_float_to_half(m / -8.0f) : 0;", "oracle_float_to_half(amax / 8.0f) : 0;")],
    "scale_over_7": [("oracle_float_to_half(m / -8.0f) : 0;", "oracle_float_to_half(m / -7.0f) : 0;")],
    "nibbles_swapped": [("(uint8_t)(q[j] | (q[j + 16] << 4))", "(uint8_t)(q[j + 16] | (q[j] << 4))")],
    "half_round_down": [("if (rest > half || (rest == half && (kept & 1u)))", "if (rest > half)")],
    "half_no_subnormals": [("        if (e == 0)\n            return sign;                       /* binary32 subnormals",
                            "        if (1)\n            return sign;                       /* binary32 subnormals")],
    "last_tie_wins": [("        if (a > amax) {", "        if (a >= amax && a > 0.0f) {")],
}


@pytest.mark.parametrize("name", sorted(QUANT_MUTATIONS))
def test_quantizer_mutation_is_caught(name, tmp_path):
    src = open(oracle.SRC).read()
    for old, new in QUANT_MUTATIONS[name]:
        assert old in src, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new)
    mdir = tmp_path / "src"
    mdir.mkdir()
    (mdir / "q4_0_oracle.c").write_text(src)
    shutil.copy(oracle.HDR, mdir / "q4_0_oracle.h")
    lib = oracle.build_library(str(mdir / "q4_0_oracle.c"), str(tmp_path / "libmut.so"), include_dir=str(mdir))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in QUANT_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutation {name}"
    os.remove(lib)
