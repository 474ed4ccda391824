"""Checks that pin the oracle to facts other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  They run against the real oracle (test_oracle_pins.py) and against
deliberately broken copies of it (test_oracle_mutations.py), which shows that
a plausible mistake anywhere in the oracle fails at least one of them.

What each pin rests on:
  nbytes          the block_q4_0 struct is 2 + 16 bytes, a row is K/32 blocks
                  ("Binding GGUF weights to the compute graph", section 2.3)
  half decode     numpy's own binary16 -> float64 conversion, all 65536 patterns
  golden blocks   hand-derived values in tests/golden/q4_0_blocks.txt
  zero point      a block of all-8 codes decodes to zeros carrying d's sign
  golden mul_mat  hand-derived sums in tests/golden/q4_0_mul_mat_small.txt
  one-hot         x = e_k selects column k of the dequantised W exactly
  brute force     tiny shapes against numpy float64 matmul of a numpy decode
  exact case      d = 2^-e and x in {1, 2, -1/2}: y is an exactly
                  representable integer sum times a power of two
"""
from __future__ import annotations

import ctypes

import numpy as np

import synth
from golden_io import read_blocks, read_mul_mat, same_f32_bits


def pin_nbytes(orc):
    class BlockQ4_0(ctypes.Structure):
        _pack_ = 1
        _fields_ = [("d", ctypes.c_uint16), ("qs", ctypes.c_uint8 * 16)]

    assert ctypes.sizeof(BlockQ4_0) == 18
    for M, K in [(1, 32), (256, 1024), (11008, 4096), (4096, 11008),
                 (32000, 4096), (14336, 4096), (3, 288)]:
        assert orc.nbytes(M, K) == M * (K // 32) * ctypes.sizeof(BlockQ4_0)
    # 7B-like layer: 4 x 4096^2 + 2 x 11008x4096 + 4096x11008 weights, 32 layers
    total = 32 * sum(orc.nbytes(M, K) for _, M, K in synth.LAYER_MATRICES)
    assert total == 3_642_753_024


def pin_half_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.half_to_float(bits).astype(np.float64)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    for h in (0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0xFBFF):
        assert orc.half_to_double(h) == float(np.uint16(h).view(np.float16))


def pin_golden_blocks(orc):
    recs = read_blocks()
    assert len(recs) >= 8
    for name, raw, values in recs:
        got = orc.dequant(raw, 1, 32)[0]
        ok = same_f32_bits(got, values)
        assert ok.all(), f"{name}: {got} != {values}"


def pin_zero_point_sign(orc):
    rng = np.random.Generator(np.random.SFC64(7))
    nb = 64
    d = rng.uniform(0.001, 100.0, nb).astype(np.float16)
    d[nb // 2:] = -d[nb // 2:]
    qs = np.full((1, nb, 16), 0x88, dtype=np.uint8)
    W = synth.blocks_from_parts(d.view(np.uint16).reshape(1, nb), qs)
    w = orc.dequant(W, 1, 32 * nb)[0].reshape(nb, 32).view(np.uint32)
    assert (w[: nb // 2] == 0x00000000).all()          # +0.0
    assert (w[nb // 2:] == 0x80000000).all()           # -0.0


def pin_golden_mul_mat(orc):
    rec = read_mul_mat()
    Y, S = orc.mul_mat(rec["W"], rec["M"], rec["K"], rec["X"])
    assert np.array_equal(Y, rec["Y"]), (Y, rec["Y"])
    assert np.array_equal(S, rec["S"]), (S, rec["S"])


def pin_one_hot(orc):
    M, K = 7, 96
    W = synth.q4_0_weights(M, K, seed=11)
    deq = orc.dequant(W, M, K)
    for k in (0, 1, 15, 16, 17, 31, 32, 63, 95):
        x = np.zeros((1, K), dtype=np.float32)
        x[0, k] = 1.0
        Y, S = orc.mul_mat(W, M, K, x)
        assert np.array_equal(Y[0], deq[:, k].astype(np.float64))
        assert np.array_equal(S[0], np.abs(deq[:, k]).astype(np.float64))


def _numpy_decode(W: np.ndarray, M: int, K: int) -> np.ndarray:
    blk = np.ascontiguousarray(W).reshape(M, K // 32, 18)
    d = blk[:, :, 0:2].copy().view("<f2")[:, :, 0].astype(np.float64)
    qs = blk[:, :, 2:].astype(np.int64)
    codes = np.concatenate([qs & 0x0F, qs >> 4], axis=2)        # [M, nb, 32]
    return (d[:, :, None] * (codes - 8)).reshape(M, K)


def pin_brute_force(orc):
    shapes = [(1, 32, 1), (3, 64, 2), (8, 96, 5), (5, 32, 8), (2, 96, 3), (7, 64, 1)]
    for i, (M, K, N) in enumerate(shapes):
        W = synth.q4_0_weights(M, K, seed=100 + i)
        X = synth.activations(N, K, seed=200 + i)
        Y, S = orc.mul_mat(W, M, K, X)
        w = _numpy_decode(W, M, K)
        x = X.astype(np.float64)
        y_ref = x @ w.T
        s_ref = np.abs(x) @ np.abs(w).T
        assert Y.shape == (N, M)
        assert np.allclose(Y, y_ref, rtol=1e-12, atol=1e-14), (M, K, N)
        assert np.allclose(S, s_ref, rtol=1e-12, atol=1e-14), (M, K, N)


def pin_exact_power_of_two(orc):
    M, K = 5, 256
    nb = K // 32
    rng = np.random.Generator(np.random.SFC64(3))
    qs = rng.integers(0, 256, (M, nb, 16), dtype=np.uint8)
    for e in (3, 5, 8):
        d = np.full((M, nb), 2.0 ** -e, dtype=np.float16)
        W = synth.blocks_from_parts(d.view(np.uint16), qs)
        X = np.stack([np.full(K, v, dtype=np.float32) for v in (1.0, 2.0, -0.5)])
        Y, _ = orc.mul_mat(W, M, K, X)
        codes = np.concatenate([qs & 0x0F, qs >> 4], axis=2).astype(np.int64) - 8
        isum = codes.reshape(M, K).sum(axis=1)                     # exact integers
        for n, v in enumerate((1.0, 2.0, -0.5)):
            assert np.array_equal(Y[n], isum * (2.0 ** -e) * v)


ALL_PINS = [pin_nbytes, pin_half_all_patterns, pin_golden_blocks, pin_zero_point_sign,
            pin_golden_mul_mat, pin_one_hot, pin_brute_force, pin_exact_power_of_two]
