"""Pins of the oracle's Q5_0 and Q5_1 functions against facts other than
themselves, and planted mistakes (in a copy of the oracle, on the CPU) that a
pin must catch.

Facts used: hand-derived blocks (tests/golden/q5_blocks.txt); the byte counts
the reading fixes (22 and 24 bytes per 32 weights); exact identities with the
independently pinned Q4_1 (a Q5_1 block whose high bits are all 0 is the
Q4_1 block with the same fields; a Q5_0 block with all high bits 0 is the Q4_1
block with m = -16 d, with all high bits 1 the one with m = 0; the test moves
the fields itself); a one-hot x selects a dequantised column; a dense fp64
matmul of the decoded weights; validation of d (and Q5_1's m)."""
import os
import shutil

import numpy as np
import pytest

import oracle
import synth
from golden_io import read_typed_blocks, same_f32_bits

Q41, Q50, Q51 = oracle.TYPE_Q4_1, oracle.TYPE_Q5_0, oracle.TYPE_Q5_1
TYPES = {"q5_0": Q50, "q5_1": Q51}


def pin_nbytes(orc):
    assert orc.type_nbytes(Q50, 11008, 4096) == 11008 * 128 * 22
    assert orc.type_nbytes(Q51, 4096, 11008) == 4096 * 344 * 24
    assert orc.type_nbytes(Q50, 3, 4096) * 8 == 3 * 4096 * 5.5     # 5.5 bits per weight
    assert orc.type_nbytes(Q51, 3, 4096) * 8 == 3 * 4096 * 6
    assert orc.type_nbytes(Q50, 3, 100) == 0


def pin_golden_blocks(orc):
    blocks = read_typed_blocks("q5_blocks.txt")
    assert len(blocks) == 4
    for tname, name, raw, values in blocks:
        assert raw.size == {"q5_0": 22, "q5_1": 24}[tname], name
        got = orc.dequant_typed(TYPES[tname], raw, 1, 32)[0]
        assert same_f32_bits(got, values).all(), f"{name}: {got} != {values}"


def _q41_from(d, m, qs):
    """Q4_1 blocks [R, nb, 20] from fp16 d, m [R, nb] and code bytes [R, nb, 16]."""
    R, nb = d.shape
    out = np.empty((R, nb, 20), dtype=np.uint8)
    out[..., 0:2] = d.astype("<f2").view(np.uint8).reshape(R, nb, 2)
    out[..., 2:4] = m.astype("<f2").view(np.uint8).reshape(R, nb, 2)
    out[..., 4:] = qs
    return out


def pin_high_bits_zero_or_one_are_q4_1(orc):
    R, K = 4, 256
    nb = K // 32
    rng = np.random.default_rng(61)
    qs = rng.integers(0, 256, (R, nb, 16)).astype(np.uint8)
    d = synth.random_scales(62, R * nb).reshape(R, nb)
    m = synth.random_scales(63, R * nb, -0.16, 0.0).reshape(R, nb)
    X = synth.activations(3, K, seed=64)
    for ones in (False, True):
        qh = np.full((R, nb, 4), 0xFF if ones else 0x00, dtype=np.uint8)
        # Q5_1, all high bits 0: Q4_1 with the same d, m, codes
        if not ones:
            W51 = np.concatenate([d.view(np.uint8).reshape(R, nb, 2), m.view(np.uint8).reshape(R, nb, 2), qh, qs],
                                 axis=-1).reshape(R, -1)
            W41 = _q41_from(d, m, qs).reshape(R, -1)
            assert same_f32_bits(orc.dequant_typed(Q51, W51, R, K), orc.dequant_typed(Q41, W41, R, K)).all()
            ya, sa = orc.mul_mat_typed(Q51, W51, R, K, X)
            yb, sb = orc.mul_mat_typed(Q41, W41, R, K, X)
            assert np.array_equal(ya, yb) and np.array_equal(sa, sb)
        # Q5_0: high bits 0 -> Q4_1 with m = -16 d (exact); high bits 1 -> m = 0
        W50 = np.concatenate([d.view(np.uint8).reshape(R, nb, 2), qh, qs], axis=-1).reshape(R, -1)
        m0 = np.zeros_like(d) if ones else (-16 * d.astype(np.float32)).astype(np.float16)
        W41 = _q41_from(d, m0, qs).reshape(R, -1)
        a = orc.dequant_typed(Q50, W50, R, K)
        b = orc.dequant_typed(Q41, W41, R, K)
        assert np.array_equal(a, b)               # +0 == -0: q = 16 with d < 0 gives -0 in Q5_0
        ya, _ = orc.mul_mat_typed(Q50, W50, R, K, X)
        yb, _ = orc.mul_mat_typed(Q41, W41, R, K, X)
        assert np.array_equal(ya, yb)


def pin_one_hot_column(orc):
    for t in (Q50, Q51):
        M, K = 9, 96
        W = synth.typed_weights(t, M, K, seed=65 + t)
        dense = orc.dequant_typed(t, W, M, K)
        for k in (0, 15, 16, 31, 32, 63, 95):
            x = np.zeros((1, K), dtype=np.float32)
            x[0, k] = 1.0
            y, _ = orc.mul_mat_typed(t, W, M, K, x)
            assert np.array_equal(y[0], dense[:, k].astype(np.float64)), (t, k)


def pin_dense_brute_force(orc):
    for t in (Q50, Q51):
        M, K, N = 4, 128, 3
        W = synth.typed_weights(t, M, K, seed=67 + t)
        X = synth.activations(N, K, seed=68)
        dense = orc.dequant_typed(t, W, M, K).astype(np.float64)
        y, s = orc.mul_mat_typed(t, W, M, K, X)
        assert np.allclose(y, X.astype(np.float64) @ dense.T, rtol=1e-12, atol=1e-12)
        assert np.allclose(s, np.abs(X.astype(np.float64)) @ np.abs(dense).T, rtol=1e-12, atol=1e-12)


def pin_validate(orc):
    M, K = 3, 128
    for t, bb in ((Q50, 22), (Q51, 24)):
        W = synth.typed_weights(t, M, K, seed=69 + t).reshape(M, 4, bb)
        W[1, 2, 0:2] = np.array([0x7C00], dtype="<u2").view(np.uint8)      # d = inf: block 6
        W[2, 3, 2:4] = np.array([0x7E00], dtype="<u2").view(np.uint8)      # Q5_1: m = NaN (block 11); Q5_0: high bits
        want = (2, 6) if t == Q51 else (1, 6)
        assert orc.validate(t, W.reshape(M, -1), M, K) == want, t


Q5_PINS = [pin_nbytes, pin_golden_blocks, pin_high_bits_zero_or_one_are_q4_1, pin_one_hot_column,
           pin_dense_brute_force, pin_validate]


@pytest.mark.parametrize("pin", Q5_PINS, ids=lambda p: p.__name__)
def test_q5_pin(pin, orc):
    pin(orc)


Q5_MUTATIONS = {
    "high_bit_order_reversed": [("int q = nib | (int)(((qh >> e) & 1u) << 4);",
                                 "int q = nib | (int)(((qh >> (31 - e)) & 1u) << 4);")],
    "high_bits_big_endian": [("uint32_t qh = (uint32_t)blk[off] | ((uint32_t)blk[off + 1] << 8) |\n"
                              "                  ((uint32_t)blk[off + 2] << 16) | ((uint32_t)blk[off + 3] << 24);",
                              "uint32_t qh = (uint32_t)blk[off + 3] | ((uint32_t)blk[off + 2] << 8) |\n"
                              "                  ((uint32_t)blk[off + 1] << 16) | ((uint32_t)blk[off] << 24);")],
    "high_half_uses_low_bits": [("int q = nib | (int)(((qh >> e) & 1u) << 4);",
                                 "int q = nib | (int)(((qh >> (e & 15)) & 1u) << 4);")],
    "zero_point_8": [("            w[e] = d * (float)(q - 16);", "            w[e] = d * (float)(q - 8);")],
    "q5_1_min_dropped": [("            w[e] = dq + m;", "            w[e] = dq;")],
    "nibbles_swapped": [("int nib = e < 16 ? (qs[e] & 0x0F) : (qs[e - 16] >> 4);",
                         "int nib = e < 16 ? (qs[e] >> 4) : (qs[e - 16] & 0x0F);")],
    "high_bit_weight_32": [("int q = nib | (int)(((qh >> e) & 1u) << 4);", "int q = nib | (int)(((qh >> e) & 1u) << 5);")],
    "q5_1_fields_at_q5_0_offset": [("int off = type == ORACLE_TYPE_Q5_1 ? 4 : 2;", "int off = 2;")],
    "q5_0_block_size_20": [("    case ORACLE_TYPE_Q5_0: return 22;", "    case ORACLE_TYPE_Q5_0: return 20;")],
    "validate_ignores_q5_1_min": [("if (type == ORACLE_TYPE_Q4_1 || type == ORACLE_TYPE_Q4_K || type == ORACLE_TYPE_Q5_1)",
                                   "if (type == ORACLE_TYPE_Q4_1 || type == ORACLE_TYPE_Q4_K)")],
}


@pytest.mark.parametrize("name", sorted(Q5_MUTATIONS))
def test_q5_mutation_is_caught(name, tmp_path):
    src = open(oracle.SRC).read()
    for old, new in Q5_MUTATIONS[name]:
        assert src.count(old) == 1, f"mutation anchor missing or ambiguous: {old!r}"
        src = src.replace(old, new)
    mdir = tmp_path / "src"
    mdir.mkdir()
    (mdir / "q4_0_oracle.c").write_text(src)
    shutil.copy(oracle.HDR, mdir / "q4_0_oracle.h")
    lib = oracle.build_library(str(mdir / "q4_0_oracle.c"), str(tmp_path / "libmut.so"), include_dir=str(mdir))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in Q5_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutation {name}"
    os.remove(lib)
