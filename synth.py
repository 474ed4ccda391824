"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA path.

This module only draws random numbers and lays them out as raw bytes; it holds
none of the Q4_0 arithmetic (no decoding, no products).  Both sides of every
parity check read the arrays it returns.

Workload shapes follow the 7B-like model on the pages ("Binding GGUF weights to the
compute graph", section 2.4: per-layer q/k/v/o, gate/up/down projections) and the
capability probe batch of 512 tokens ("GGUF loading, mmap and tensor placement",
step six).  Value distributions:

* ``qs``: uniform random bytes (all 256 values, so every 4-bit code appears);
* ``d``: fp16 (round-to-nearest-even) of U[0.005, 0.02] drawn in fp64;
* activations: fp32 N(0, 1).

Random bits come from numpy's SFC64 generator (``random_raw``), whose output
stream is fixed by its published definition, so the same seed yields the same
bytes on x86-64 and aarch64.
"""
from __future__ import annotations

import numpy as np

QK4_0 = 32           # weights per block_q4_0
BLOCK_BYTES = 18     # ggml_half d (2 bytes) + uint8_t qs[16]

# Matrix ids inside one 7B-like layer, in graph order.
LAYER_MATRICES = (
    ("attn_q", 4096, 4096),
    ("attn_k", 4096, 4096),
    ("attn_v", 4096, 4096),
    ("attn_output", 4096, 4096),
    ("ffn_gate", 11008, 4096),
    ("ffn_up", 11008, 4096),
    ("ffn_down", 4096, 11008),
)
N_LAYERS = 32


def seed_for(workload: int, matrix: int, layer: int = 0) -> int:
    """Seed of one matrix of one workload (stable across runs)."""
    return 0x51A00000 + 16 * workload + matrix + 1000 * layer


def _raw_u64(seed: int, n_words: int) -> np.ndarray:
    return np.random.SFC64(seed).random_raw(n_words)


def random_bytes(seed: int, n: int) -> np.ndarray:
    words = _raw_u64(seed, (n + 7) // 8)
    return words.view(np.uint8)[:n]


def random_scales(seed: int, n: int, lo: float = 0.005, hi: float = 0.02) -> np.ndarray:
    """n fp16 scales: round-to-nearest-even of U[lo, hi] drawn in fp64."""
    rng = np.random.Generator(np.random.SFC64(seed ^ 0x5CA1E))
    u = rng.random(n, dtype=np.float64) * (hi - lo) + lo
    return u.astype("<f2")


def q4_0_weights(M: int, K: int, seed: int, d_range=(0.005, 0.02)) -> np.ndarray:
    """A Q4_0 weight matrix with M rows of K weights, as raw bytes.

    Shape ``[M, K/32*18]`` uint8: row m is K/32 consecutive 18-byte blocks, each
    the little-endian fp16 scale (RNE of U[d_range] drawn in fp64) followed by
    16 bytes of packed codes.
    """
    if K % QK4_0:
        raise ValueError("K must be a multiple of 32")
    nb = K // QK4_0
    out = np.empty((M, nb, BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 2:] = random_bytes(seed, M * nb * 16).reshape(M, nb, 16)
    out[:, :, 0:2] = random_scales(seed, M * nb, *d_range).view(np.uint8).reshape(M, nb, 2)
    return out.reshape(M, nb * BLOCK_BYTES)


def activations(N: int, K: int, seed: int) -> np.ndarray:
    """fp32 N(0,1) activations, shape [N, K] (K innermost, as ggml ne[0])."""
    rng = np.random.Generator(np.random.SFC64(seed ^ 0xAC7))
    return rng.standard_normal((N, K), dtype=np.float32)


def blocks_from_parts(d_bits: np.ndarray, qs: np.ndarray) -> np.ndarray:
    """Assemble blocks from explicit fp16 bit patterns and code bytes.

    ``d_bits``: uint16 ``[M, nb]``; ``qs``: uint8 ``[M, nb, 16]``.  Returns the
    ``[M, nb*18]`` byte matrix.  Used for hand-built edge cases.
    """
    d_bits = np.asarray(d_bits, dtype="<u2")
    qs = np.asarray(qs, dtype=np.uint8)
    M, nb = d_bits.shape
    out = np.empty((M, nb, BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = d_bits.view(np.uint8).reshape(M, nb, 2)
    out[:, :, 2:] = qs
    return out.reshape(M, nb * BLOCK_BYTES)


def expert_ids(T: int, S: int, E: int, seed: int, skew: float = 0.0) -> np.ndarray:
    """int32 [T, S] expert ids: each token picks S distinct experts out of E
    (S <= E), as a top-S router does.  skew = 0 draws them uniformly; skew > 0
    weights expert e by 1 / (e + 1)**skew (Zipf-like: a few experts take most
    tokens), sampled without replacement by Efraimidis-Spirakis keys u**(1/w)."""
    if not 0 < S <= E:
        raise ValueError("need 0 < S <= E")
    rng = np.random.Generator(np.random.SFC64(seed ^ 0x1D5))
    u = rng.random((T, E), dtype=np.float64)
    w = 1.0 / np.power(np.arange(1, E + 1, dtype=np.float64), skew)
    keys = np.power(u, 1.0 / w)
    return np.argsort(-keys, axis=1, kind="stable")[:, :S].astype(np.int32)


def moe_weights(E: int, M: int, K: int, seed: int) -> np.ndarray:
    """E Q4_0 matrices of M rows each, one after the other: [E*M, K/32*18]."""
    return np.concatenate([q4_0_weights(M, K, seed + 7919 * e) for e in range(E)], axis=0)


def q4_k_weights(M: int, K: int, seed: int, d_scale: float = 1.0) -> np.ndarray:
    """Q4_K weights as raw bytes [M, K/256*144]: per 256-weight super-block a
    little-endian fp16 d ~ U[1e-4, 2e-4] and fp16 dmin ~ U[7.5e-4, 1.5e-3]
    (RNE of fp64 draws, times d_scale), then 12 random bytes (every pattern
    is a valid set of 6-bit sub-block scales and mins) and 128 random code
    bytes.  With sub-block scales and mins uniform on 0..63, dmin ~ 7.5 d
    centres the weights d*sc*q - dmin*m roughly on zero, as a quantiser that
    fits each sub-block's range would."""
    if K % 256:
        raise ValueError("K must be a multiple of 256")
    nb = K // 256
    out = np.empty((M, nb, 144), dtype=np.uint8)
    out[:, :, 4:] = random_bytes(seed, M * nb * 140).reshape(M, nb, 140)
    out[:, :, 0:2] = random_scales(seed, M * nb, 1e-4 * d_scale, 2e-4 * d_scale).view(np.uint8).reshape(M, nb, 2)
    out[:, :, 2:4] = random_scales(seed ^ 0x4D19, M * nb, 7.5e-4 * d_scale,
                                   1.5e-3 * d_scale).view(np.uint8).reshape(M, nb, 2)
    return out.reshape(M, nb * 144)


def typed_weights(qtype: int, M: int, K: int, seed: int, d_scale: float = 1.0) -> np.ndarray:
    """Weights in one of the block formats, as raw bytes [M, K/32*bytes]:
    0 = Q4_0 (q4_0_weights), 1 = Q4_1 (fp16 d ~ U[0.005, 0.02], fp16 m ~
    U[-0.16, 0], 16 random code bytes), 2 = Q8_0 (fp16 d ~ U[0.0003, 0.0012],
    32 random int8 code bytes), 3 = Q4_K (q4_k_weights: [M, K/256*144]), 4 / 5 =
    Q5_0 / Q5_1 (fp16 d ~ U[0.0025, 0.01], Q5_1 also m ~ U[-0.16, 0], 20 random
    bytes of high bits and codes).
    Scales are RNE fp16 of values drawn in fp64; d_scale multiplies the ranges
    of d and m (e.g. 100 for O(1) weights)."""
    if qtype == 0:
        return q4_0_weights(M, K, seed, (0.005 * d_scale, 0.02 * d_scale))
    if qtype == 3:
        return q4_k_weights(M, K, seed, d_scale)
    if qtype in (4, 5):
        # Q5_0 / Q5_1: fp16 d ~ U[0.0025, 0.01] (half Q4_0's range: codes span 32
        # levels), Q5_1 also fp16 m ~ U[-0.16, 0]; 4 random high-bit bytes and 16
        # random code bytes
        if K % QK4_0:
            raise ValueError("K must be a multiple of 32")
        nb = K // QK4_0
        bb = 22 if qtype == 4 else 24
        out = np.empty((M, nb, bb), dtype=np.uint8)
        out[:, :, bb - 20:] = random_bytes(seed, M * nb * 20).reshape(M, nb, 20)
        out[:, :, 0:2] = random_scales(seed, M * nb, 0.0025 * d_scale, 0.01 * d_scale).view(np.uint8).reshape(M, nb, 2)
        if qtype == 5:
            out[:, :, 2:4] = random_scales(seed ^ 0x3117, M * nb, -0.16 * d_scale, 0.0).view(np.uint8).reshape(M, nb, 2)
        return out.reshape(M, nb * bb)
    if K % QK4_0:
        raise ValueError("K must be a multiple of 32")
    nb = K // QK4_0
    if qtype == 1:
        out = np.empty((M, nb, 20), dtype=np.uint8)
        out[:, :, 4:] = random_bytes(seed, M * nb * 16).reshape(M, nb, 16)
        out[:, :, 0:2] = random_scales(seed, M * nb, 0.005 * d_scale, 0.02 * d_scale).view(np.uint8).reshape(M, nb, 2)
        out[:, :, 2:4] = random_scales(seed ^ 0x3117, M * nb, -0.16 * d_scale, 0.0).view(np.uint8).reshape(M, nb, 2)
        return out.reshape(M, nb * 20)
    if qtype == 2:
        out = np.empty((M, nb, 34), dtype=np.uint8)
        out[:, :, 2:] = random_bytes(seed, M * nb * 32).reshape(M, nb, 32)
        out[:, :, 0:2] = random_scales(seed, M * nb, 0.0003 * d_scale, 0.0012 * d_scale).view(np.uint8).reshape(M, nb, 2)
        return out.reshape(M, nb * 34)
    raise ValueError("unknown block type")


def wide_range_activations(N: int, K: int, seed: int, tokens, magnitudes=(1e5, 1e9)) -> np.ndarray:
    """fp32 N(0, 1) activations whose listed tokens carry, in a quarter of their
    32-element blocks (at least one), values scaled by 10^U[log10 lo, log10 hi]
    (beyond the fp16 range): the wide-range stress input of the decode path."""
    X = activations(N, K, seed)
    rng = np.random.Generator(np.random.SFC64(seed + 1))
    lo, hi = np.log10(magnitudes[0]), np.log10(magnitudes[1])
    nb = K // QK4_0
    for n in tokens:
        blocks = rng.choice(nb, size=max(1, nb // 4), replace=False)
        for b in blocks:
            X[n, b * QK4_0:(b + 1) * QK4_0] *= np.float32(10.0 ** rng.uniform(lo, hi))
    return X
