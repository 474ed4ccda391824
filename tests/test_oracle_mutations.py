"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins catch every one of them.  This is what makes the pins evidence: a
dropped term, a wrong sign, index, nibble order or transposed operand in the
oracle would not survive them."""
import os
import shutil

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTATIONS = {
    "nibble_order_swapped": [("int q_lo = qs[j] & 0x0F;", "int q_lo = qs[j] >> 4;"),
                             ("int q_hi = qs[j] >> 4;", "int q_hi = qs[j] & 0x0F;")],
    "interleaved_nibbles": [("w[b * QK + j] = ", "w[b * QK + 2 * j] = "),
                            ("w[b * QK + j + 16] = ", "w[b * QK + 2 * j + 1] = ")],
    "zero_point_7": [("(float)(q_lo - 8)", "(float)(q_lo - 7)"),
                     ("(float)(q_hi - 8)", "(float)(q_hi - 7)")],
    "factored_form_loses_negative_zero": [
        ("d * (float)(q_lo - 8)", "(d * (float)q_lo - 8.0f * d)"),
        ("d * (float)(q_hi - 8)", "(d * (float)q_hi - 8.0f * d)")],
    "scale_big_endian": [("blk[0] | (blk[1] << 8)", "blk[1] | (blk[0] << 8)")],
    "half_exponent_bias": [("e - 25", "e - 24")],
    "half_subnormal_scale": [("ldexp((double)f, -24)", "ldexp((double)f, -25)")],
    "half_implicit_one_dropped": [("(double)(1024 + f)", "(double)(f)")],
    "last_code_byte_dropped": [("for (int j = 0; j < 16; ++j)", "for (int j = 0; j < 15; ++j)")],
    "x_transposed": [("double p = (double)w[k] * (double)x[k];",
                      "double p = (double)w[k] * (double)X[(size_t)k * (size_t)N + (size_t)n % (size_t)(N > 0 ? N : 1)];")],
    "y_transposed": [("Y[(size_t)n * (size_t)M + (size_t)m] = acc;",
                      "Y[(size_t)m * (size_t)N + (size_t)n] = acc;")],
    "abs_sum_signed": [("acc_abs += fabs(p);", "acc_abs += p;")],
    "sign_of_product": [("acc += p;", "acc -= p;")],
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    src = open(oracle.SRC).read()
    for old, new in MUTATIONS[name]:
        assert old in src, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new)
    mdir = tmp_path / "src"
    mdir.mkdir()
    (mdir / "q4_0_oracle.c").write_text(src)
    shutil.copy(oracle.HDR, mdir / "q4_0_oracle.h")
    lib = oracle.build_library(str(mdir / "q4_0_oracle.c"), str(tmp_path / "libmut.so"),
                               include_dir=str(mdir))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutation {name}"
    os.remove(lib)
