"""Q4_1 and Q8_0 on the GPU against the oracle: dequantisation bit for bit,
MUL_MAT within |y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-5 (fp64 oracle)."""
import numpy as np
import pytest

import oracle
import synth
from golden_io import read_typed_blocks, same_f32_bits
from gpu_util import assert_mul_mat_close, cores

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import quantized_block_q4_gb300 as gq
else:  # collected on CPU machines, never run there (marked gpu)
    gq = None

TYPES = [1, 2]  # GQ_TYPE_Q4_1, GQ_TYPE_Q8_0 (same numbering as oracle.TYPE_*)
NAMES = {1: "q4_1", 2: "q8_0"}


def dev(a):
    return torch.from_numpy(np.array(a, copy=True)).cuda()


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K", [(256, 1024), (11008, 4096), (4096, 11008), (1, 32), (7, 96), (129, 288), (300, 8192)])
def test_dequant_bit_exact(qtype, M, K):
    W = synth.typed_weights(qtype, M, K, seed=13000 + M + K + qtype)
    got = gq.dequant(qtype, dev(W), K).cpu().numpy()
    assert same_f32_bits(got, oracle.get().dequant_typed(qtype, W, M, K)).all()


def test_dequant_golden_blocks():
    for tname, name, raw, values in read_typed_blocks():
        qtype = {"q4_1": 1, "q8_0": 2}[tname]
        got = gq.dequant(qtype, dev(raw), 32).cpu().numpy()[0]
        assert same_f32_bits(got, values).all(), name


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
def test_dequant_unaligned(qtype):
    M, K = 37, 320
    W = synth.typed_weights(qtype, M, K, seed=13100 + qtype)
    buf = torch.zeros(W.size + 16, dtype=torch.uint8, device="cuda")
    buf[3:3 + W.size] = dev(W.reshape(-1))
    out = torch.full((M * K + 1,), float("nan"), device="cuda")
    gq.gq_dequant(qtype, buf.data_ptr() + 3, M, K, out.data_ptr() + 4)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.isnan(got[0])
    assert same_f32_bits(got[1:].reshape(M, K), oracle.get().dequant_typed(qtype, W, M, K)).all()


def check(qtype, M, K, N, seed, sample=None):
    W = synth.typed_weights(qtype, M, K, seed)
    X = synth.activations(N, K, seed + 1)
    y = gq.mul_mat(qtype, dev(W), dev(X)).cpu().numpy()
    rows = np.arange(M) if sample is None else np.random.default_rng(seed).choice(M, sample, replace=False)
    row_bytes = K // 32 * gq.TYPE_BLOCK_BYTES[qtype]
    Wr = W.reshape(M, row_bytes)[rows]
    y_ref, s_ref = oracle.get().mul_mat_typed(qtype, Wr, len(rows), K, X, nthreads=cores())
    return assert_mul_mat_close(y[:, rows], y_ref, s_ref, f"{NAMES[qtype]} M={M} K={K} N={N}")


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K,N", [(256, 1024, 1), (300, 512, 3), (129, 96, 4), (77, 288, 5), (64, 4096, 16),
                                   (33, 1024, 33), (1, 32, 1)])
def test_mul_mat_matches_oracle(qtype, M, K, N):
    check(qtype, M, K, N, seed=13200 + M + K + N + qtype)


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K,N", [(11008, 4096, 1), (4096, 11008, 1), (11008, 4096, 8), (14336, 4096, 512),
                                   (4096, 11008, 512), (32000, 4096, 16)])
def test_mul_mat_full_size_sampled_rows(qtype, M, K, N):
    check(qtype, M, K, N, seed=13300 + N + qtype, sample=48)


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K,N", [(300, 512, 16), (129, 1024, 100), (1000, 2048, 257), (64, 256, 128), (700, 4096, 2),
                                   (130, 768, 5)])
def test_tensor_core_path_matches_oracle(qtype, M, K, N):
    """N >= 16 with K % 256 == 0: the tcgen05 kernel with this block format
    (several row tiles, ragged M and N, one and several 256-k chunks)."""
    check(qtype, M, K, N, seed=13600 + M + N + qtype)


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
def test_tensor_core_and_scalar_paths_agree(qtype):
    """The same N = 32 product through the tensor-core kernel and through the
    scalar kernel (GQ_OPT_FORCE_GENERIC), both against the oracle."""
    M, K, N = 500, 1024, 32
    check(qtype, M, K, N, seed=13700 + qtype)
    gq.gq_set_option(gq.GQ_OPT_FORCE_GENERIC, 1)
    try:
        check(qtype, M, K, N, seed=13700 + qtype)
    finally:
        gq.gq_set_option(gq.GQ_OPT_FORCE_GENERIC, 0)


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
def test_mul_mat_unaligned(qtype):
    M, K, N = 40, 256, 3
    W = synth.typed_weights(qtype, M, K, seed=13400 + qtype)
    X = synth.activations(N, K, 13401)
    wb = torch.zeros(W.size + 8, dtype=torch.uint8, device="cuda")
    wb[1:1 + W.size] = dev(W.reshape(-1))
    xb = torch.zeros(N * K + 1, device="cuda")
    xb[1:] = dev(X).reshape(-1)
    Y = torch.empty(N, M, device="cuda")
    gq.gq_mul_mat(qtype, wb.data_ptr() + 1, M, K, xb.data_ptr() + 4, N, Y)
    torch.cuda.synchronize()
    y_ref, s_ref = oracle.get().mul_mat_typed(qtype, W, M, K, X)
    assert_mul_mat_close(Y.cpu().numpy(), y_ref, s_ref, "unaligned")


def test_typed_errors_and_q4_0_dispatch():
    L = gq._lib
    assert L.gq_mul_mat(7, None, 4, 32, None, 1, None, None) == gq.GQ_ERR_SHAPE
    assert L.gq_dequant(7, None, 4, 32, None, None) == gq.GQ_ERR_SHAPE
    assert L.gq_type_nbytes(2, 3, 64) == 3 * 2 * 34 and L.gq_type_nbytes(9, 3, 64) == 0
    M, K, N = 100, 512, 2
    W = synth.q4_0_weights(M, K, seed=13500)
    X = synth.activations(N, K, 13501)
    a = gq.mul_mat(0, dev(W), dev(X))
    b = gq.mul_mat_q4_0(dev(W), dev(X))
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K", [(256, 1024), (1000, 4096), (33, 256), (4096, 11008)])
def test_decode_kernel_and_scalar_agree(qtype, M, K):
    """N = 1 through the mma.sync decode kernel (20- or 34-byte blocks) and
    through the scalar kernel (GQ_OPT_FORCE_GENERIC), both against the oracle,
    with and without the weights-static / x-static promises (which select the
    4-warp CTA)."""
    seed = 13800 + M + K + qtype
    check(qtype, M, K, 1, seed, sample=None if M <= 1000 else 64)
    for flag in (gq.GQ_OPT_WEIGHTS_STATIC, gq.GQ_OPT_X_STATIC):
        gq.gq_set_option(flag, 1)
    try:
        check(qtype, M, K, 1, seed, sample=None if M <= 1000 else 64)
    finally:
        for flag in (gq.GQ_OPT_WEIGHTS_STATIC, gq.GQ_OPT_X_STATIC):
            gq.gq_set_option(flag, 0)
    gq.gq_set_option(gq.GQ_OPT_FORCE_GENERIC, 1)
    try:
        check(qtype, M, K, 1, seed, sample=None if M <= 1000 else 64)
    finally:
        gq.gq_set_option(gq.GQ_OPT_FORCE_GENERIC, 0)


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("N", [2, 7, 9, 15])
def test_small_batch_decode_kernel(qtype, N):
    """2..15 tokens with K % 256 == 0: the mma.sync decode kernel (one or two
    n8 token tiles), ragged rows, K over several x chunks."""
    check(qtype, 1000, 8192, N, seed=13900 + N + qtype)
