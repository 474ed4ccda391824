"""Pins of the oracle's Q4_0 quantiser against facts other than itself.

The quantiser follows the block-quantisation formula of "Architecture and
module overview" (weight-loading section): q(w) = clip(round(w/s) + z, q_min,
q_max), w_hat = s*(q - z), with the error model E[e] ~ 0, Var(e) ~ Delta^2/12
for Delta = s.  For Q4_0: z = 8, q in [0, 15], the fp16 scale d is s.  The
pages leave the choice of s open; the reading pinned here is d =
binary16(m / -8) for the weight m of largest magnitude (the first on ties).

Each pin takes an oracle object and raises AssertionError on a violation.
"""
from __future__ import annotations

import numpy as np


def _blocks(q: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """uint8 [rows, K/32*18] -> (d bits [rows, nb], codes [rows, nb, 32])."""
    rows = q.shape[0]
    b = q.reshape(rows, -1, 18)
    d = b[..., 0].astype(np.uint16) | (b[..., 1].astype(np.uint16) << 8)
    qs = b[..., 2:]
    codes = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)
    return d, codes


def pin_float_to_half_matches_numpy(orc):
    """binary32 -> binary16 rounding (nearest even) against numpy's conversion,
    on values across the whole binary16 range, its subnormals, exact ties and
    overflow."""
    rng = np.random.default_rng(11)
    vals = [rng.standard_normal(3000).astype(np.float32) * np.float32(s)
            for s in (1e-8, 3e-6, 6e-5, 1e-3, 1.0, 1e3, 6e4)]
    # exact binary16 ties: halfway between neighbouring binary16 values
    h = rng.integers(0, 0x7BFF, 3000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float32)
    hi = (h + 1).view(np.float16).astype(np.float32)
    ties = ((lo.astype(np.float64) + hi.astype(np.float64)) / 2).astype(np.float32)
    extra = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
                      2.0 ** -25 * 1.0000001, 2.0 ** -26, 6.1035156e-05, np.inf, -np.inf], dtype=np.float32)
    allv = np.concatenate(vals + [ties, -ties, extra])
    got = np.array([orc.float_to_half(v) for v in allv], dtype=np.uint16)
    with np.errstate(over="ignore"):
        ref = allv.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} binary16 roundings differ from numpy"
    nan = orc.float_to_half(float("nan"))
    assert (nan & 0x7C00) == 0x7C00 and (nan & 0x3FF) != 0, "NaN must stay NaN"


def pin_round_trip_is_exact(orc):
    """Dequantising a block with a code 0 (weight -8d, the unique largest
    magnitude) and quantising again gives the same bytes: the scale is
    recovered exactly and every w/d is an integer."""
    rng = np.random.default_rng(12)
    rows, K = 64, 256
    q = rng.integers(0, 256, (rows, K // 32, 18)).astype(np.uint8)
    d = (rng.uniform(0.005, 0.02, (rows, K // 32)) * rng.choice([-1, 1], (rows, K // 32)))
    dbits = d.astype(np.float16).view(np.uint16)
    q[..., 0] = dbits & 0xFF
    q[..., 1] = dbits >> 8
    q[..., 2 + rng.integers(0, 16, (rows, K // 32))[..., None] * 0] &= 0xF0  # element 0 of each block: code 0
    blocks = q.reshape(rows, -1)
    w = orc.dequant(blocks, rows, K)
    again = orc.quantize(w)
    assert np.array_equal(again, blocks), "quantise(dequantise(B)) != B"


def pin_codes_are_nearest_levels(orc):
    """Every code is the level d*(q-8), q in [0, 15], nearest to its weight,
    by brute force over the 16 levels in fp64 (up to ties)."""
    rng = np.random.default_rng(13)
    w = rng.standard_normal((16, 1024)).astype(np.float32)
    qb = orc.quantize(w)
    dbits, codes = _blocks(qb)
    d = dbits.astype(np.uint16).view(np.float16).astype(np.float64)[..., None]
    wb = w.reshape(16, -1, 32).astype(np.float64)
    levels = d[..., None] * (np.arange(16, dtype=np.float64) - 8)           # [r, b, 1, 16]
    err = np.abs(wb[..., None] - levels)                                     # [r, b, 32, 16]
    chosen = np.take_along_axis(err, codes[..., None].astype(np.int64), axis=-1)[..., 0]
    best = err.min(axis=-1)
    assert np.all(chosen <= best + 1e-6 * np.abs(d)), "a code is not the nearest level"


def pin_scale_from_largest_magnitude(orc):
    """d is binary16(m / -8) for the weight m of largest magnitude (numpy
    argmax picks the first on ties, as the reading says)."""
    rng = np.random.default_rng(14)
    w = (rng.standard_normal((8, 512)) * 3).astype(np.float32)
    dbits, _ = _blocks(orc.quantize(w))
    wb = w.reshape(8, -1, 32)
    idx = np.abs(wb).argmax(axis=-1)
    m = np.take_along_axis(wb, idx[..., None], axis=-1)[..., 0]
    with np.errstate(over="ignore"):
        ref = (m / np.float32(-8)).astype(np.float16).view(np.uint16)
    assert np.array_equal(dbits, ref), "the scale is not binary16(m / -8)"


def pin_error_model(orc):
    """Uniform data: |e| <= Delta/2 for every element that is not clipped, the
    mean error ~ 0 and Var(e)/Delta^2 ~ 1/12 (the pages' error model)."""
    rng = np.random.default_rng(15)
    w = rng.uniform(-1, 1, (64, 4096)).astype(np.float32)
    qb = orc.quantize(w)
    dbits, codes = _blocks(qb)
    d = dbits.view(np.float16).astype(np.float64)[..., None]
    what = d * (codes.astype(np.float64) - 8)
    e = what - w.reshape(64, -1, 32).astype(np.float64)
    delta = np.abs(d)
    # m maps to -8 and |w| <= |m|, so w/d >= -8; only w/d > 7.5 (opposite-sign
    # weights near the extreme) is clipped, to 15.  The model describes the
    # rounding errors of the others.
    inner = (w.reshape(64, -1, 32).astype(np.float64) / d) <= 7.5
    assert np.all(np.abs(e[inner]) <= np.broadcast_to(delta, e.shape)[inner] * 0.5 * (1 + 1e-6)), "|e| > Delta/2"
    assert np.all(codes[~inner] == 15), "a clipped element does not get code 15"
    r = (e / delta)[inner]
    assert abs(r.mean()) < 0.01, f"mean error {r.mean():.4f} Delta, expected ~0"
    assert abs(r.var() - 1 / 12) < 0.05 / 12, f"Var(e)/Delta^2 = {r.var():.5f}, expected ~1/12"
    assert np.count_nonzero(~inner) < 0.05 * inner.size, "too many clipped elements"


def pin_special_blocks(orc):
    """All-zero block: d = 0 and every code 8.  One nonzero weight v: d =
    binary16(v/-8), its code 0, every other code 8."""
    w = np.zeros((1, 64), dtype=np.float32)
    w[0, 32 + 5] = 3.0       # second block: element 5
    w[0, 32 + 20] = 0.0
    qb = orc.quantize(w)
    assert qb[0, :18].tobytes() == bytes([0, 0]) + bytes([0x88] * 16), "all-zero block"
    dbits, codes = _blocks(qb)
    assert dbits[0, 1] == np.float16(3.0 / -8).view(np.uint16)
    expect = np.full(32, 8)
    expect[5] = 0
    assert np.array_equal(codes[0, 1], expect), f"one-hot block codes {codes[0, 1]}"
    # a negative extreme: its code is 0 as well (d > 0)
    w2 = np.zeros((1, 32), dtype=np.float32)
    w2[0, 17] = -2.0
    dbits2, codes2 = _blocks(orc.quantize(w2))
    assert dbits2[0, 0] == np.float16(0.25).view(np.uint16) and codes2[0, 0, 17] == 0
    # a tie in magnitude: the first of +3 (element 2) and -3 (element 7) sets
    # d = -3/8, so element 2 gets code 0 and element 7 (w/d = 8) clips to 15
    w3 = np.zeros((1, 32), dtype=np.float32)
    w3[0, 2], w3[0, 7], w3[0, 9] = 3.0, -3.0, 0.75
    dbits3, codes3 = _blocks(orc.quantize(w3))
    assert dbits3[0, 0] == np.float16(-0.375).view(np.uint16), "the first weight of largest magnitude sets d"
    assert codes3[0, 0, 2] == 0 and codes3[0, 0, 7] == 15 and codes3[0, 0, 9] == 6


QUANT_PINS = [pin_float_to_half_matches_numpy, pin_round_trip_is_exact, pin_codes_are_nearest_levels,
              pin_scale_from_largest_magnitude, pin_error_model, pin_special_blocks]
