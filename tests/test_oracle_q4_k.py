"""Pins of the oracle's Q4_K functions against facts other than themselves,
and planted mistakes (in a copy of the oracle, on the CPU) that a pin must
catch.

Facts used:
  * hand-derived super-blocks (tests/golden/q4_k_blocks.txt), whose bytes were
    packed by hand from chosen fields;
  * the byte count the reading fixes: ne[0]/256 super-blocks of 144 bytes per
    row (4.5 bits per weight), nothing for K % 256 != 0;
  * an exact identity with Q4_1, whose own pins are independent: with d and
    dmin powers of two, d*sc_j and -dmin*m_j are exact fp16 numbers, so
    sub-block j decodes exactly like a Q4_1 block with those as its d and m and
    the same codes; the test packs the 6-bit fields and moves the codes between
    the two layouts itself;
  * closed forms (all codes 0: w = -dmin*m_j; m = 0: w = d*sc_j*q);
  * a one-hot x selects a dequantised column; a dense fp64 matmul of the
    decoded weights on tiny shapes;
  * validation flags exactly the super-blocks with a non-finite d or dmin.
"""
import os
import shutil

import numpy as np
import pytest

import oracle
import synth
from golden_io import read_typed_blocks, same_f32_bits

Q4K, Q41 = oracle.TYPE_Q4_K, oracle.TYPE_Q4_1


def pack_fields(sc, m):
    """The 12 bytes holding 6-bit sub-block scales sc[0..7] and mins m[0..7]
    (the reading in q4_0_oracle.h), written from the field description."""
    sc = np.asarray(sc, dtype=np.int64)
    m = np.asarray(m, dtype=np.int64)
    out = np.zeros(sc.shape[:-1] + (12,), dtype=np.int64)
    for j in range(4):
        out[..., j] = (sc[..., j] & 63) | ((sc[..., j + 4] >> 4) << 6)
        out[..., 4 + j] = (m[..., j] & 63) | ((m[..., j + 4] >> 4) << 6)
        out[..., 8 + j] = (sc[..., j + 4] & 15) | ((m[..., j + 4] & 15) << 4)
    return out.astype(np.uint8)


def q4_k_from_fields(d_bits, dmin_bits, sc, m, codes):
    """Super-blocks [R, nb, 144] from fp16 bit patterns [R, nb], fields [R, nb, 8]
    and codes [R, nb, 256] (code of weight i of the super-block)."""
    R, nb = d_bits.shape
    out = np.empty((R, nb, 144), dtype=np.uint8)
    out[..., 0:2] = np.asarray(d_bits, dtype="<u2").view(np.uint8).reshape(R, nb, 2)
    out[..., 2:4] = np.asarray(dmin_bits, dtype="<u2").view(np.uint8).reshape(R, nb, 2)
    out[..., 4:16] = pack_fields(sc, m)
    c = np.asarray(codes, dtype=np.uint8).reshape(R, nb, 4, 64)
    out[..., 16:] = (c[..., :32] | (c[..., 32:] << 4)).reshape(R, nb, 128)
    return out


def pin_nbytes(orc):
    assert orc.type_nbytes(Q4K, 11008, 4096) == 11008 * 16 * 144
    assert orc.type_nbytes(Q4K, 4096, 11008) == 4096 * 43 * 144                # 11008 = 43 * 256
    assert orc.type_nbytes(Q4K, 3, 4096) * 8 == 3 * 4096 * 4.5          # 4.5 bits per weight
    assert orc.type_nbytes(Q4K, 3, 4096 + 32) == 0                         # K must be a multiple of 256
    assert orc.type_nbytes(Q4K, 0, 4096) == 0


def pin_golden_blocks(orc):
    blocks = [b for b in read_typed_blocks("q4_k_blocks.txt") if b[0] == "q4_k"]
    assert len(blocks) == 4
    for _, name, raw, values in blocks:
        assert raw.size == 144 and values.size == 256, name
        got = orc.dequant_typed(Q4K, raw, 1, 256)[0]
        assert same_f32_bits(got, values).all(), f"{name}: first mismatch at {np.argmin(same_f32_bits(got, values))}"


def _subblocks_as_q4_1(seed, R, nb):
    """Random Q4_K super-blocks whose d, dmin are powers of two, and the Q4_1
    blocks that must decode identically (8 per super-block, in order)."""
    rng = np.random.default_rng(seed)
    e_d = rng.integers(-14, -3, (R, nb))
    e_m = rng.integers(-14, -3, (R, nb))
    sign = rng.integers(0, 2, (R, nb))
    d = np.ldexp(1.0, e_d) * np.where(sign == 1, -1.0, 1.0)
    dmin = np.ldexp(1.0, e_m)
    sc = rng.integers(0, 64, (R, nb, 8))
    m = rng.integers(0, 64, (R, nb, 8))
    codes = rng.integers(0, 16, (R, nb, 256))
    W = q4_k_from_fields(d.astype(np.float16).view(np.uint16), dmin.astype(np.float16).view(np.uint16), sc, m, codes)
    # Q4_1 block j of a super-block: d1 = d*sc_j, m1 = -dmin*m_j (exact fp16), element i = code of weight 32j + i
    d1 = (d[..., None] * sc).astype(np.float16)
    m1 = (-dmin[..., None] * m).astype(np.float16)
    assert np.array_equal(d1.astype(np.float64), d[..., None] * sc)    # exactness of the identity's premise
    assert np.array_equal(m1.astype(np.float64), -dmin[..., None] * m)
    cj = codes.reshape(R, nb, 8, 32).astype(np.uint8)
    W1 = np.empty((R, nb, 8, 20), dtype=np.uint8)
    W1[..., 0:2] = d1.view(np.uint8).reshape(R, nb, 8, 2)
    W1[..., 2:4] = m1.view(np.uint8).reshape(R, nb, 8, 2)
    W1[..., 4:] = cj[..., :16] | (cj[..., 16:] << 4)
    return W.reshape(R, nb * 144), W1.reshape(R, nb * 8 * 20)


def pin_subblocks_are_q4_1(orc):
    R, nb = 5, 3
    K = 256 * nb
    W, W1 = _subblocks_as_q4_1(51, R, nb)
    a = orc.dequant_typed(Q4K, W, R, K)
    b = orc.dequant_typed(Q41, W1, R, K)
    assert same_f32_bits(a, b).all()
    X = synth.activations(3, K, seed=52)
    yk, sk = orc.mul_mat_typed(Q4K, W, R, K, X)
    y1, s1 = orc.mul_mat_typed(Q41, W1, R, K, X)
    assert np.array_equal(yk, y1) and np.array_equal(sk, s1)


def pin_closed_forms(orc):
    rng = np.random.default_rng(53)
    R, nb = 2, 2
    d = rng.uniform(0.01, 0.1, (R, nb)).astype(np.float16)
    dmin = rng.uniform(0.01, 0.1, (R, nb)).astype(np.float16)
    sc = rng.integers(0, 64, (R, nb, 8))
    m = rng.integers(0, 64, (R, nb, 8))
    zero = np.zeros((R, nb, 256), dtype=np.int64)
    W = q4_k_from_fields(d.view(np.uint16), dmin.view(np.uint16), sc, m, zero)
    got = orc.dequant_typed(Q4K, W, R, 256 * nb).reshape(R, nb, 8, 32)
    want = -(dmin.astype(np.float64)[..., None] * m)                      # every code 0
    assert np.array_equal(got.astype(np.float64), np.repeat(want[..., None], 32, axis=-1))
    codes = rng.integers(0, 16, (R, nb, 256))
    W = q4_k_from_fields(d.view(np.uint16), dmin.view(np.uint16), sc, np.zeros_like(m), codes)
    got = orc.dequant_typed(Q4K, W, R, 256 * nb).reshape(R, nb, 8, 32)
    want = d.astype(np.float64)[..., None, None] * sc[..., None] * codes.reshape(R, nb, 8, 32)   # every min 0
    assert np.array_equal(got.astype(np.float64), want)


def pin_one_hot_column(orc):
    M, K = 7, 512
    W = synth.q4_k_weights(M, K, seed=54)
    dense = orc.dequant_typed(Q4K, W, M, K)
    for k in (0, 31, 32, 63, 64, 200, 255, 256, 511):
        x = np.zeros((1, K), dtype=np.float32)
        x[0, k] = 1.0
        y, _ = orc.mul_mat_typed(Q4K, W, M, K, x)
        assert np.array_equal(y[0], dense[:, k].astype(np.float64)), k


def pin_dense_brute_force(orc):
    M, K, N = 4, 512, 3
    W = synth.q4_k_weights(M, K, seed=55)
    X = synth.activations(N, K, seed=56)
    dense = orc.dequant_typed(Q4K, W, M, K).astype(np.float64)
    y, s = orc.mul_mat_typed(Q4K, W, M, K, X)
    assert np.allclose(y, X.astype(np.float64) @ dense.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(s, np.abs(X.astype(np.float64)) @ np.abs(dense).T, rtol=1e-12, atol=1e-12)


def pin_validate(orc):
    M, K = 4, 1024
    W = synth.q4_k_weights(M, K, seed=57).reshape(M, 4, 144)
    assert orc.validate(Q4K, W.reshape(M, -1), M, K) == (0, None)
    W[1, 2, 2:4] = np.array([0x7C00], dtype="<u2").view(np.uint8)        # dmin = +inf in super-block 1*4 + 2
    W[3, 0, 0:2] = np.array([0x7E00], dtype="<u2").view(np.uint8)        # d = NaN in super-block 12
    W[3, 1, 4:16] = 0xFF                                                  # 6-bit fields: any pattern is valid
    assert orc.validate(Q4K, W.reshape(M, -1), M, K) == (2, 6)


Q4K_PINS = [pin_nbytes, pin_golden_blocks, pin_subblocks_are_q4_1, pin_closed_forms, pin_one_hot_column,
            pin_dense_brute_force, pin_validate]


@pytest.mark.parametrize("pin", Q4K_PINS, ids=lambda p: p.__name__)
def test_q4_k_pin(pin, orc):
    pin(orc)


Q4K_MUTATIONS = {
    "scale_and_min_swapped": [("        sc[j] = b[j] & 0x3F;\n        m[j] = b[4 + j] & 0x3F;",
                               "        sc[j] = b[4 + j] & 0x3F;\n        m[j] = b[j] & 0x3F;")],
    "high_bits_from_wrong_byte": [("sc[4 + j] = (b[8 + j] & 0x0F) | ((b[j] >> 6) << 4);",
                                   "sc[4 + j] = (b[8 + j] & 0x0F) | ((b[4 + j] >> 6) << 4);")],
    "high_bits_dropped": [("m[4 + j] = (b[8 + j] >> 4) | ((b[4 + j] >> 6) << 4);", "m[4 + j] = (b[8 + j] >> 4);")],
    "nibble_fields_swapped": [("sc[4 + j] = (b[8 + j] & 0x0F)", "sc[4 + j] = (b[8 + j] >> 4)"),
                              ("m[4 + j] = (b[8 + j] >> 4)", "m[4 + j] = (b[8 + j] & 0x0F)")],
    "min_added": [("w[64 * c + l] = dl * (float)q_lo - ml;", "w[64 * c + l] = dl * (float)q_lo + ml;")],
    "d_and_dmin_swapped": [("    float d = le_half_at(blk);\n    float dmin = le_half_at(blk + 2);",
                            "    float d = le_half_at(blk + 2);\n    float dmin = le_half_at(blk);")],
    "nibbles_swapped": [("int q_lo = qs[32 * c + l] & 0x0F;\n            int q_hi = qs[32 * c + l] >> 4;",
                         "int q_lo = qs[32 * c + l] >> 4;\n            int q_hi = qs[32 * c + l] & 0x0F;")],
    "high_nibble_same_subblock": [("int jl = 2 * c, jh = 2 * c + 1;", "int jl = 2 * c, jh = 2 * c;")],
    "codes_start_early": [("const uint8_t *qs = blk + 16;", "const uint8_t *qs = blk + 12;")],
    "codes_interleaved": [("w[64 * c + 32 + l] = dh * (float)q_hi - mh;", "w[64 * c + 32 + (l ^ 1)] = dh * (float)q_hi - mh;")],
    "block_bytes_128": [("    case ORACLE_TYPE_Q4_K: return 144;", "    case ORACLE_TYPE_Q4_K: return 128;")],
    "zero_point_8": [("w[64 * c + l] = dl * (float)q_lo - ml;", "w[64 * c + l] = dl * (float)(q_lo - 8) - ml;")],
    "validate_ignores_dmin": [("if (type == ORACLE_TYPE_Q4_1 || type == ORACLE_TYPE_Q4_K || type == ORACLE_TYPE_Q5_1)",
                               "if (type == ORACLE_TYPE_Q4_1 || type == ORACLE_TYPE_Q5_1)")],
}


@pytest.mark.parametrize("name", sorted(Q4K_MUTATIONS))
def test_q4_k_mutation_is_caught(name, tmp_path):
    src = open(oracle.SRC).read()
    for old, new in Q4K_MUTATIONS[name]:
        assert src.count(old) == 1, f"mutation anchor missing or ambiguous: {old!r}"
        src = src.replace(old, new)
    mdir = tmp_path / "src"
    mdir.mkdir()
    (mdir / "q4_0_oracle.c").write_text(src)
    shutil.copy(oracle.HDR, mdir / "q4_0_oracle.h")
    lib = oracle.build_library(str(mdir / "q4_0_oracle.c"), str(tmp_path / "libmut.so"), include_dir=str(mdir))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in Q4K_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutation {name}"
    os.remove(lib)
