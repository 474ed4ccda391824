"""Pins of the oracle's row-data validation (CPU only).

A block is invalid when one of its fp16 scale fields (d; for Q4_1 also m) is
NaN or infinite ("GGUF loading, mmap and tensor placement", the section on
--check-tensors: ggml_validate_row_data checks each row's scales and integers);
codes are never invalid.  Pinned against numpy's float16 classification of
all 65,536 bit patterns (an independent decoder), hand-placed bad blocks at
known positions, and the empty cases.
"""
import os
import shutil

import numpy as np
import pytest

import oracle

Q4_0, Q4_1, Q8_0 = oracle.TYPE_Q4_0, oracle.TYPE_Q4_1, oracle.TYPE_Q8_0
BB = oracle.BLOCK_BYTES


def one_block_rows(qtype, d_bits, m_bits=None, code_byte=0x00):
    """One block per row: row i has scale bits d_bits[i] (and m_bits[i])."""
    n = len(d_bits)
    W = np.full((n, BB[qtype]), code_byte, dtype=np.uint8)
    W[:, 0] = d_bits & 0xFF
    W[:, 1] = d_bits >> 8
    if qtype == Q4_1:
        mb = np.zeros(n, dtype=np.uint16) if m_bits is None else m_bits
        W[:, 2] = mb & 0xFF
        W[:, 3] = mb >> 8
    return W


def numpy_finite(bits):
    return np.isfinite(np.asarray(bits, dtype=np.uint16).view(np.float16))


def pin_every_fp16_pattern_as_scale(o):
    bits = np.arange(65536, dtype=np.uint16)
    bad = np.flatnonzero(~numpy_finite(bits))
    for qtype in (Q4_0, Q4_1, Q8_0):
        count, first = o.validate(qtype, one_block_rows(qtype, bits), 65536, 32)
        assert count == len(bad) == 2048          # exponent 31: two infinities and 2,046 NaNs
        assert first == bad[0] == 0x7C00


def pin_single_patterns_against_numpy(o):
    rng = np.random.Generator(np.random.SFC64(91))
    picks = np.concatenate([rng.integers(0, 65536, 300), [0x0000, 0x8000, 0x0001, 0x7BFF, 0xFBFF, 0x7C00,
                                                           0xFC00, 0x7C01, 0x7E00, 0xFFFF, 0x3C00]])
    for qtype in (Q4_0, Q4_1, Q8_0):
        for p in picks.astype(np.uint16):
            count, first = o.validate(qtype, one_block_rows(qtype, np.array([p], np.uint16)), 1, 32)
            expect_bad = not numpy_finite([p])[0]
            assert count == int(expect_bad) and (first == 0 if expect_bad else first is None), hex(int(p))


def pin_q4_1_min_field_is_checked_too(o):
    one = np.array([0x3C00], np.uint16)
    for m, bad in ((0x3C00, False), (0x7C00, True), (0xFE00, True), (0x0001, False)):
        W = one_block_rows(Q4_1, one, np.array([m], np.uint16))
        assert o.validate(Q4_1, W, 1, 32) == ((1, 0) if bad else (0, None)), hex(m)
    # a non-finite min is not a problem for Q4_0, whose bytes 2..3 are codes
    W = one_block_rows(Q4_0, one)
    W[0, 2:4] = [0x00, 0x7C]
    assert o.validate(Q4_0, W, 1, 32) == (0, None)


def pin_codes_never_make_a_block_invalid(o):
    for qtype in (Q4_0, Q4_1, Q8_0):
        for code in (0x00, 0x7F, 0x80, 0xFF):
            W = one_block_rows(qtype, np.array([0x3C00, 0x0400], np.uint16), code_byte=code)
            assert o.validate(qtype, W, 2, 32) == (0, None)


def pin_planted_bad_blocks_count_and_first(o):
    M, K = 7, 320                      # 10 blocks per row
    nb = K // 32
    for qtype in (Q4_0, Q4_1, Q8_0):
        W = np.zeros((M, nb, BB[qtype]), dtype=np.uint8)
        W[:, :, 1] = 0x3C              # d = 1.0 everywhere
        planted = [(2, 9), (5, 0), (6, 3)]
        for r, b in planted:
            W[r, b, 1] = 0x7E          # d = NaN
        count, first = o.validate(qtype, W.reshape(M, -1), M, K)
        assert count == len(planted)
        assert first == 2 * nb + 9


def pin_empty_matrices(o):
    assert o.validate(Q4_0, np.zeros(0, np.uint8), 0, 64) == (0, None)
    assert o.validate(Q4_1, np.zeros(0, np.uint8), 5, 0) == (0, None)


PINS = [pin_every_fp16_pattern_as_scale, pin_single_patterns_against_numpy, pin_q4_1_min_field_is_checked_too,
        pin_codes_never_make_a_block_invalid, pin_planted_bad_blocks_count_and_first, pin_empty_matrices]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.get())


# Plausible mistakes in a copy of the oracle's validation, each caught by a pin.
MUTATIONS = {
    "nan_not_detected": [("int bad = !isfinite(oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8))));",
                          "int bad = isinf(oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8))));")],
    "q4_1_min_ignored": [("if (type == ORACLE_TYPE_Q4_1 || type == ORACLE_TYPE_Q4_K || type == ORACLE_TYPE_Q5_1)   /* m, or dmin */\n            bad |=",
                          "if (type == ORACLE_TYPE_Q4_K || type == ORACLE_TYPE_Q5_1)\n            bad |=")],
    "first_is_the_last": [("if (*count == 0)\n                *first = b;", "*first = b;")],
    "q4_0_block_stride": [("const uint8_t *blk = W + b * (uint64_t)bb;", "const uint8_t *blk = W + b * 18u;")],
    "scale_big_endian": [("int bad = !isfinite(oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8))));",
                          "int bad = !isfinite(oracle_half_to_double((uint16_t)(blk[1] | (blk[0] << 8))));")],
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
    lib = oracle.build_library(str(mdir / "q4_0_oracle.c"), str(tmp_path / "libmut.so"), include_dir=str(mdir))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutation {name}"
    os.remove(lib)
