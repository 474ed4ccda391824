"""The CUDA quantiser (gq_quantize_q4_0) against the oracle, byte for byte.

The codes are integers decided by an fp32 quotient and the scale by a
binary16 rounding, so both sides must agree exactly (see the oracle's
quantize_block and include/gq.h for the rule)."""
import numpy as np
import pytest
import torch

import oracle
import quantized_block_q4_gb300 as gq
import synth

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_quantize(W: np.ndarray) -> np.ndarray:
    q = gq.quantize_q4_0(dev(W.astype(np.float32)))
    torch.cuda.synchronize()
    return q.cpu().numpy()


def check(W: np.ndarray, label: str):
    got = gpu_quantize(W)
    ref = oracle.get().quantize(W)
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        r, c = bad[0]
        raise AssertionError(f"{label}: {len(bad)} bytes differ, first at row {r} byte {c}: "
                             f"{got[r, c // 18 * 18:(c // 18 + 1) * 18].tobytes().hex()} vs "
                             f"{ref[r, c // 18 * 18:(c // 18 + 1) * 18].tobytes().hex()}")


@pytest.mark.parametrize("M,K", [(256, 1024), (11008, 4096), (4096, 11008), (14336, 4096), (1, 32), (3, 96),
                                 (129, 256), (7, 288)])
def test_quantize_matches_oracle(M, K):
    rng = np.random.default_rng(8000 + M + K)
    W = rng.standard_normal((M, K)).astype(np.float32) * np.float32(0.05)
    check(W, f"{M}x{K} normal")


def test_quantize_value_ranges():
    """Blocks whose scale is a binary16 subnormal, a large normal, or overflows
    to infinity; mixed signs and magnitudes within blocks."""
    rng = np.random.default_rng(8100)
    M, K = 64, 2048
    W = rng.standard_normal((M, K)).astype(np.float64)
    scales = 10.0 ** rng.uniform(-9, 6, (M, K // 32, 1))
    W = (W.reshape(M, -1, 32) * scales).reshape(M, K).astype(np.float32)
    W[0, :32] = 1e30 * rng.standard_normal(32)      # d overflows binary16 -> +-inf
    W[1, :32] = 3e-7 * rng.standard_normal(32)      # d is a binary16 subnormal
    check(W, "value ranges")


def test_quantize_special_blocks():
    W = np.zeros((1, 32 * 8), dtype=np.float32)
    W[0, 32 + 5] = 3.0                               # one nonzero
    W[0, 64 + 2], W[0, 64 + 7] = 3.0, -3.0           # tie: the first wins
    W[0, 96:128] = -0.0                              # negative zeros: an all-zero block
    W[0, 128:160] = np.linspace(-1, 1, 32)
    W[0, 128 + 4] = np.nan                           # NaN weight: code 8
    W[0, 160:192] = np.linspace(-2, 2, 32)
    W[0, 160 + 9] = np.inf                           # inf weight: d = -inf, codes 8
    W[0, 192:224] = 1.0                              # all equal: d = -1/8, every code 0
    W[0, 224:256] = np.arange(32) - 16.0
    check(W, "special blocks")
    # the same blocks in whole warps of 32 blocks (the coalesced-load path),
    # one row of 64 blocks and four rows of 16
    check(np.tile(W, (1, 8)), "special blocks, whole warps")
    check(np.tile(W, (4, 2)), "special blocks, four rows")


def test_quantize_unaligned_pointers():
    M, K = 33, 512
    rng = np.random.default_rng(8200)
    W = rng.standard_normal((M, K)).astype(np.float32)
    ref = oracle.get().quantize(W)
    src = torch.zeros(M * K + 1, dtype=torch.float32, device="cuda")
    src[1:] = dev(W).reshape(-1)                     # 4-byte but not 16-byte aligned input
    out = torch.zeros(ref.size + 3, dtype=torch.uint8, device="cuda")
    gq.gq_quantize_q4_0(src[1:], M, K, out[3:])      # output at an odd byte offset
    torch.cuda.synchronize()
    gq.gq_sync_status()
    o = out.cpu().numpy()
    assert np.array_equal(o[3:].reshape(ref.shape), ref)
    assert not o[:3].any(), "bytes before the output were written"


def test_quantize_round_trip_on_device():
    """quantise(dequantise(B)) == B for blocks holding a code 0, entirely on the GPU."""
    M, K = 512, 4096
    W = synth.q4_0_weights(M, K, seed=8300).reshape(M, -1, 18).copy()
    W[..., 2] &= 0xF0                                # element 0 of every block: code 0
    Wd = dev(W.reshape(M, -1))
    back = gq.quantize_q4_0(gq.dequant_q4_0(Wd, K))
    torch.cuda.synchronize()
    assert torch.equal(back, Wd)


def test_quantize_argument_errors():
    L = gq._lib
    assert L.gq_quantize_q4_0(None, 4, 33, None, None) == gq.GQ_ERR_SHAPE
    assert L.gq_quantize_q4_0(None, -1, 32, None, None) == gq.GQ_ERR_SHAPE
    assert L.gq_quantize_q4_0(None, 4, 32, None, None) == gq.GQ_ERR_NULL
    assert L.gq_quantize_q4_0(None, 0, 32, None, None) == gq.GQ_OK
