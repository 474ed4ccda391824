"""Pins of the oracle's Q4_1 and Q8_0 functions against facts other than
themselves, and planted mistakes (in a copy of the oracle, on the CPU) that a
pin must catch.

Facts used: hand-derived blocks (tests/golden/legacy_blocks.txt); the byte
counts the block sizes fix; exact identities with Q4_0, whose own pins are
independent (a Q4_1 block with m = -8d decodes like the Q4_0 block with the
same d and codes; a Q8_0 block with codes in -8..7 like the Q4_0 block with
codes + 8); a one-hot x selects a dequantised column; a dense fp64 matmul of
the decoded weights on tiny shapes."""
import os
import shutil

import numpy as np
import pytest

import oracle
import synth
from golden_io import read_typed_blocks, same_f32_bits

Q40, Q41, Q80 = oracle.TYPE_Q4_0, oracle.TYPE_Q4_1, oracle.TYPE_Q8_0
TYPES = {"q4_1": Q41, "q8_0": Q80}


def pin_nbytes(orc):
    assert orc.type_nbytes(Q41, 11008, 4096) == 11008 * 128 * 20
    assert orc.type_nbytes(Q80, 4096, 11008) == 4096 * 344 * 34
    assert orc.type_nbytes(Q40, 7, 64) == orc.nbytes(7, 64)


def pin_golden_blocks(orc):
    for tname, name, raw, values in read_typed_blocks():
        got = orc.dequant_typed(TYPES[tname], raw, 1, 32)[0]
        assert same_f32_bits(got, values).all(), f"{name}: {got} != {values}"


def pin_q4_1_with_min_minus_8d_is_q4_0(orc):
    M, K = 6, 256
    W0 = synth.q4_0_weights(M, K, seed=31).reshape(M, -1, 18)
    d = W0[..., 0:2].copy().view(np.float16)
    m = (-8 * d.astype(np.float32)).astype(np.float16)        # exact: d times a power of two
    W1 = np.empty((M, K // 32, 20), dtype=np.uint8)
    W1[..., 0:2] = W0[..., 0:2]
    W1[..., 2:4] = m.view(np.uint8)
    W1[..., 4:] = W0[..., 2:]
    a = orc.dequant_typed(Q41, W1.reshape(M, -1), M, K)
    b = orc.dequant(W0.reshape(M, -1), M, K)
    assert np.array_equal(a, b)                                # +0 == -0: only q = 8 with d < 0 differs in sign
    X = synth.activations(3, K, seed=32)
    y1, s1 = orc.mul_mat_typed(Q41, W1.reshape(M, -1), M, K, X)
    y0, s0 = orc.mul_mat(W0.reshape(M, -1), M, K, X)
    assert np.array_equal(y1, y0) and np.array_equal(s1, s0)


def pin_q8_0_small_codes_are_q4_0(orc):
    M, K = 5, 128
    rng = np.random.default_rng(33)
    codes = rng.integers(-8, 8, (M, K // 32, 32))
    d = synth.random_scales(34, M * K // 32).reshape(M, K // 32)
    W8 = np.empty((M, K // 32, 34), dtype=np.uint8)
    W8[..., 0:2] = d.view(np.uint8).reshape(M, K // 32, 2)
    W8[..., 2:] = (codes & 0xFF).astype(np.uint8)
    u = (codes + 8).astype(np.uint8)
    W4 = np.empty((M, K // 32, 18), dtype=np.uint8)
    W4[..., 0:2] = W8[..., 0:2]
    W4[..., 2:] = u[..., :16] | (u[..., 16:] << 4)
    assert same_f32_bits(orc.dequant_typed(Q80, W8.reshape(M, -1), M, K), orc.dequant(W4.reshape(M, -1), M, K)).all()
    X = synth.activations(2, K, seed=35)
    y8, s8 = orc.mul_mat_typed(Q80, W8.reshape(M, -1), M, K, X)
    y4, s4 = orc.mul_mat(W4.reshape(M, -1), M, K, X)
    assert np.array_equal(y8, y4) and np.array_equal(s8, s4)


def pin_one_hot_column(orc):
    for t in (Q41, Q80):
        M, K = 9, 96
        W = synth.typed_weights(t, M, K, seed=36 + t)
        dense = orc.dequant_typed(t, W, M, K)
        for k in (0, 17, 31, 32, 95):
            x = np.zeros((1, K), dtype=np.float32)
            x[0, k] = 1.0
            y, _ = orc.mul_mat_typed(t, W, M, K, x)
            assert np.array_equal(y[0], dense[:, k].astype(np.float64)), (t, k)


def pin_dense_brute_force(orc):
    for t in (Q41, Q80):
        M, K, N = 4, 64, 3
        W = synth.typed_weights(t, M, K, seed=40 + t)
        X = synth.activations(N, K, seed=41)
        dense = orc.dequant_typed(t, W, M, K).astype(np.float64)
        y, s = orc.mul_mat_typed(t, W, M, K, X)
        assert np.allclose(y, X.astype(np.float64) @ dense.T, rtol=1e-12, atol=1e-12)
        assert np.allclose(s, np.abs(X.astype(np.float64)) @ np.abs(dense).T, rtol=1e-12, atol=1e-12)


LEGACY_PINS = [pin_nbytes, pin_golden_blocks, pin_q4_1_with_min_minus_8d_is_q4_0, pin_q8_0_small_codes_are_q4_0,
               pin_one_hot_column, pin_dense_brute_force]


@pytest.mark.parametrize("pin", LEGACY_PINS, ids=lambda p: p.__name__)
def test_legacy_pin(pin, orc):
    pin(orc)


LEGACY_MUTATIONS = {
    "q4_1_min_first": [("float m = le_half(blk + 2);", "float m = le_half(blk);"),
                       ("float d = le_half(blk);\n        if (type == ORACLE_TYPE_Q4_1)",
                        "float d = le_half(blk + (type == ORACLE_TYPE_Q4_1 ? 2 : 0));\n        if (type == ORACLE_TYPE_Q4_1)")],
    "q4_1_no_min": [("                wb[j] = lo + m;", "                wb[j] = lo;")],
    "q4_1_zero_point": [("float lo = d * (float)(qs[j] & 0x0F);", "float lo = d * (float)((qs[j] & 0x0F) - 8);")],
    "q4_1_nibbles_swapped": [("float lo = d * (float)(qs[j] & 0x0F);\n                float hi = d * (float)(qs[j] >> 4);",
                              "float lo = d * (float)(qs[j] >> 4);\n                float hi = d * (float)(qs[j] & 0x0F);")],
    "q4_1_fields_after_codes": [("const uint8_t *qs = blk + 4;", "const uint8_t *qs = blk + 2;")],
    "q8_0_unsigned_codes": [("int q = qs[j] < 128 ? (int)qs[j] : (int)qs[j] - 256;", "int q = (int)qs[j];")],
    "q8_0_sign_flipped": [("                wb[j] = d * (float)q;", "                wb[j] = -d * (float)q;")],
    "q8_0_block_size_32": [("    case ORACLE_TYPE_Q8_0: return 34;", "    case ORACLE_TYPE_Q8_0: return 33;")],
    "typed_mul_mat_drops_last_k": [("            for (int64_t k = 0; k < K; ++k) {\n                double p = (double)w[k] * (double)x[k];\n                acc += p;\n                acc_abs += fabs(p);\n            }\n            Y[(size_t)n * (size_t)M + (size_t)m] = acc;\n            S[(size_t)n * (size_t)M + (size_t)m] = acc_abs;\n        }\n        free(w);\n    }\n}\n",
                                    "            for (int64_t k = 0; k + 1 < K; ++k) {\n                double p = (double)w[k] * (double)x[k];\n                acc += p;\n                acc_abs += fabs(p);\n            }\n            Y[(size_t)n * (size_t)M + (size_t)m] = acc;\n            S[(size_t)n * (size_t)M + (size_t)m] = acc_abs;\n        }\n        free(w);\n    }\n}\n")],
}


@pytest.mark.parametrize("name", sorted(LEGACY_MUTATIONS))
def test_legacy_mutation_is_caught(name, tmp_path):
    src = open(oracle.SRC).read()
    for old, new in LEGACY_MUTATIONS[name]:
        assert src.count(old) >= 1, f"mutation anchor missing: {old!r}"
        if name == "typed_mul_mat_drops_last_k":
            idx = src.rindex(old)                      # the typed mul_mat is the last such loop
            src = src[:idx] + new + src[idx + len(old):]
        else:
            src = src.replace(old, new)
    mdir = tmp_path / "src"
    mdir.mkdir()
    (mdir / "q4_0_oracle.c").write_text(src)
    shutil.copy(oracle.HDR, mdir / "q4_0_oracle.h")
    lib = oracle.build_library(str(mdir / "q4_0_oracle.c"), str(tmp_path / "libmut.so"), include_dir=str(mdir))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in LEGACY_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutation {name}"
    os.remove(lib)
