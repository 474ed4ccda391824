"""The repacked Q4_0 layout (gq_prepare_q4_0) and MUL_MAT on it: the layout
byte for byte, and the product against the oracle on the original weights
for K that is not a multiple of 256 (the fast kernels' box width)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_mul_mat_close, cores

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import quantized_block_q4_gb300 as gq
else:  # collected on CPU machines, never run there (marked gpu)
    gq = None


def dev(a):
    return torch.from_numpy(np.array(a, copy=True)).cuda()


def expected_layout(W, M, K):
    """Rows padded with zero blocks (00 00 then sixteen 0x88) to a multiple of 8 blocks."""
    nb, nbp = K // 32, (K + 255) // 256 * 8
    out = np.empty((M, nbp, 18), dtype=np.uint8)
    out[:, :, 0:2] = 0
    out[:, :, 2:] = 0x88
    out[:, :nb] = W.reshape(M, nb, 18)
    return out.reshape(M, nbp * 18)


@pytest.mark.parametrize("M,K", [(5, 32), (7, 96), (33, 288), (64, 1024), (3, 2880), (17, 4160)])
def test_prepare_layout(M, K):
    W = synth.q4_0_weights(M, K, seed=14000 + M + K)
    got = gq.prepare_q4_0(dev(W), K).cpu().numpy()
    assert got.shape == (M, gq.gq_prepared_q4_0_nbytes(1, K))
    assert np.array_equal(got, expected_layout(W, M, K))


def test_prepare_strided_unaligned_source():
    M, K, stride = 9, 416, 13 * 18 + 10        # rows padded by 10 bytes (ggml nb[1] > K/32*18)
    W = synth.q4_0_weights(M, K, seed=14100)
    buf = np.full(3 + M * stride, 0xEE, dtype=np.uint8)
    for r in range(M):
        buf[3 + r * stride: 3 + r * stride + W.shape[1]] = W[r]
    src = dev(buf)
    out = torch.empty((M, gq.gq_prepared_q4_0_nbytes(1, K)), dtype=torch.uint8, device="cuda")
    gq.gq_prepare_q4_0(src.data_ptr() + 3, M, K, stride, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), expected_layout(W, M, K))


def check(M, K, N, seed):
    W = synth.q4_0_weights(M, K, seed)
    X = synth.activations(N, K, seed + 1)
    Wp = gq.prepare_q4_0(dev(W), K)
    y = gq.mul_mat_q4_0_prepared(Wp, dev(X)).cpu().numpy()
    y_ref, s_ref = oracle.get().mul_mat(W, M, K, X, nthreads=cores())
    return assert_mul_mat_close(y, y_ref, s_ref, f"prepared M={M} K={K} N={N}")


@pytest.mark.parametrize("K", [96, 288, 1056, 2880, 4160])
@pytest.mark.parametrize("N", [1, 3, 8, 15, 16, 100, 512])
def test_prepared_mul_mat_matches_oracle(K, N):
    check(300 if N < 100 else 200, K, N, seed=14200 + K + N)


def test_prepared_full_size_odd_k():
    """A 11008 x 2880 matrix (2880 = 11.25 x 256) at N = 1 and N = 512: every row checked at N = 1, a
    sample of rows at N = 512."""
    M, K = 11008, 2880
    W = synth.q4_0_weights(M, K, seed=14300)
    Wp = gq.prepare_q4_0(dev(W), K)
    for N in (1, 512):
        X = synth.activations(N, K, 14301 + N)
        y = gq.mul_mat_q4_0_prepared(Wp, dev(X)).cpu().numpy()
        rows = np.arange(M) if N == 1 else np.random.default_rng(N).choice(M, 64, replace=False)
        y_ref, s_ref = oracle.get().mul_mat(W[rows], len(rows), K, X, nthreads=cores())
        assert_mul_mat_close(y[:, rows], y_ref, s_ref, f"11008 x 2880, N={N}")


@pytest.mark.parametrize("N", [1, 8, 64])
def test_prepared_equals_plain_when_k_is_whole_boxes(N):
    """K % 256 == 0: the prepared layout is the packed one, so the results match bit for bit."""
    M, K = 777, 1024
    W = dev(synth.q4_0_weights(M, K, seed=14400))
    X = dev(synth.activations(N, K, 14401))
    a = gq.mul_mat_q4_0_prepared(gq.prepare_q4_0(W, K), X)
    b = gq.mul_mat_q4_0(W, X)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_prepare_errors():
    L = gq._lib
    assert L.gq_prepare_q4_0(None, 4, 33, 0, None, None) == gq.GQ_ERR_SHAPE
    assert L.gq_prepare_q4_0(None, 4, 64, 20, None, None) == gq.GQ_ERR_SHAPE   # stride shorter than a row (36)
    assert L.gq_prepare_q4_0(None, 4, 64, 0, None, None) == gq.GQ_ERR_NULL
    assert L.gq_prepared_q4_0_nbytes(3, 288) == 3 * 2 * 144 and L.gq_prepared_q4_0_nbytes(1, 33) == 0
