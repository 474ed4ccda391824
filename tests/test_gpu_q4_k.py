"""Q4_K on the GPU against the oracle: dequantisation bit for bit (every
weight is d*sc_j*q - dmin*m_j rounded once to fp32), MUL_MAT within
|y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-5 (fp64 oracle) on each path: the
mma.sync decode kernel (N < 16), the tcgen05 kernel (N >= 16) and the scalar
kernel (unaligned pointers, GQ_OPT_FORCE_GENERIC); validation of d and dmin.
Inputs: synth.q4_k_weights (random 6-bit fields and codes, fp16 d ~
U[1e-4, 2e-4], dmin ~ U[7.5e-4, 1.5e-3]) and N(0, 1) activations."""
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

Q4K = 3  # GQ_TYPE_Q4_K == oracle.TYPE_Q4_K


def dev(a):
    return torch.from_numpy(np.array(a, copy=True)).cuda()


def _with_options(opts, fn):
    old = {k: gq.gq_get_option(k) for k in opts}
    try:
        for k, v in opts.items():
            gq.gq_set_option(k, v)
        return fn()
    finally:
        for k, v in old.items():
            gq.gq_set_option(k, v)


@pytest.mark.parametrize("M,K", [(1, 256), (7, 512), (129, 1280), (256, 4096), (4096, 11008), (11008, 4096)])
def test_dequant_bit_exact(M, K):
    W = synth.q4_k_weights(M, K, seed=18000 + M + K)
    got = gq.dequant(Q4K, dev(W), K).cpu().numpy()
    assert same_f32_bits(got, oracle.get().dequant_typed(Q4K, W, M, K)).all()


def test_dequant_golden_blocks():
    blocks = [b for b in read_typed_blocks("q4_k_blocks.txt") if b[0] == "q4_k"]
    assert blocks
    for _, name, raw, values in blocks:
        got = gq.dequant(Q4K, dev(raw), 256).cpu().numpy()[0]
        assert same_f32_bits(got, values).all(), name


@pytest.mark.parametrize("w_off,o_off", [(3, 4), (8, 0), (0, 4)])
def test_dequant_unaligned(w_off, o_off):
    M, K = 19, 768
    W = synth.q4_k_weights(M, K, seed=18100 + w_off)
    buf = torch.zeros(W.size + 16, dtype=torch.uint8, device="cuda")
    buf[w_off:w_off + W.size] = dev(W.reshape(-1))
    out = torch.full((M * K + 4,), float("nan"), device="cuda")
    gq.gq_dequant(Q4K, buf.data_ptr() + w_off, M, K, out.data_ptr() + o_off)
    torch.cuda.synchronize()
    gq.gq_sync_status()
    got = out.cpu().numpy()[o_off // 4:o_off // 4 + M * K]
    assert same_f32_bits(got.reshape(M, K), oracle.get().dequant_typed(Q4K, W, M, K)).all()


def check(M, K, N, seed, sample=None, d_scale=1.0, x_scale=1.0):
    W = synth.q4_k_weights(M, K, seed, d_scale)
    X = synth.activations(N, K, seed + 1) * np.float32(x_scale)
    y = gq.mul_mat(Q4K, dev(W), dev(X)).cpu().numpy()
    gq.gq_sync_status()
    rows = np.arange(M) if sample is None else np.sort(np.random.default_rng(seed).choice(M, sample, replace=False))
    Wr = W.reshape(M, K // 256 * 144)[rows]
    y_ref, s_ref = oracle.get().mul_mat_typed(Q4K, Wr, len(rows), K, X, nthreads=cores())
    return assert_mul_mat_close(y[:, rows], y_ref, s_ref, f"q4_k M={M} K={K} N={N}")


@pytest.mark.parametrize("M,K,N", [(256, 1024, 1), (300, 512, 3), (129, 256, 4), (77, 768, 5), (1000, 8192, 8),
                                   (33, 2048, 12), (500, 4096, 15), (1, 256, 1)])
def test_decode_kernel_matches_oracle(M, K, N):
    """N < 16, K % 256 == 0, aligned: the mma.sync decode kernel on 144-byte
    super-blocks (one and two n8 token tiles, ragged rows, one and several
    super-blocks and x chunks)."""
    check(M, K, N, seed=18200 + M + K + N)


@pytest.mark.parametrize("static", [0, 1])
@pytest.mark.parametrize("M,K", [(11008, 4096), (4096, 11008), (4096, 4096)])
def test_decode_sweep_shapes(M, K, static):
    """N = 1 on the sweep's shapes, with and without the weights-static and
    x-static promises (the 8-warp and the co-resident 4-warp CTA)."""
    opts = {gq.GQ_OPT_WEIGHTS_STATIC: static, gq.GQ_OPT_X_STATIC: static}
    _with_options(opts, lambda: check(M, K, 1, seed=18300 + M + static, sample=96))


@pytest.mark.parametrize("M,K,N", [(300, 512, 16), (129, 1024, 100), (1000, 2048, 257), (64, 256, 128),
                                   (700, 4096, 64), (130, 768, 17)])
def test_tensor_core_path_matches_oracle(M, K, N):
    """N >= 16: the tcgen05 kernel with Q4_K super-blocks (several row tiles,
    ragged M and N, one and several 256-k chunks, split and whole tiles)."""
    check(M, K, N, seed=18400 + M + N)


@pytest.mark.parametrize("M,K,N", [(14336, 4096, 512), (4096, 11008, 512), (32000, 4096, 16), (11008, 4096, 1),
                                   (32000, 4096, 1)])
def test_full_size_sampled_rows(M, K, N):
    check(M, K, N, seed=18500 + N, sample=48)


def test_tensor_core_decode_and_scalar_paths_agree():
    """One product through the three kernels: N = 32 tensor-core and scalar;
    N = 8 decode and scalar; each against the oracle."""
    for N in (32, 8):
        check(500, 1024, N, seed=18600 + N)
        _with_options({gq.GQ_OPT_FORCE_GENERIC: 1}, lambda: check(500, 1024, N, seed=18600 + N))


def test_mul_mat_unaligned():
    M, K, N = 40, 512, 3
    W = synth.q4_k_weights(M, K, seed=18700)
    X = synth.activations(N, K, 18701)
    wb = torch.zeros(W.size + 8, dtype=torch.uint8, device="cuda")
    wb[1:1 + W.size] = dev(W.reshape(-1))
    xb = torch.zeros(N * K + 1, device="cuda")
    xb[1:] = dev(X).reshape(-1)
    Y = torch.empty(N, M, device="cuda")
    gq.gq_mul_mat(Q4K, wb.data_ptr() + 1, M, K, xb.data_ptr() + 4, N, Y)
    torch.cuda.synchronize()
    gq.gq_sync_status()
    y_ref, s_ref = oracle.get().mul_mat_typed(Q4K, W, M, K, X)
    assert_mul_mat_close(Y.cpu().numpy(), y_ref, s_ref, "unaligned")


@pytest.mark.parametrize("N", [1, 4, 12])
def test_decode_small_x(N):
    """Activations ~ 1e-6 * N(0, 1) with O(1) weights (d and dmin x 1000):
    the decode kernel's power-of-two staging keeps the precision."""
    check(600, 4096, N, seed=18800 + N, d_scale=1000.0, x_scale=1e-6)


@pytest.mark.parametrize("N", [1, 20])
def test_large_x(N):
    """Activations ~ 1e5 * N(0, 1): fp16 staging would overflow without the
    power-of-two scaling (decode); bf16 has fp32's range (tensor core)."""
    check(300, 2048, N, seed=18900 + N, x_scale=1e5)


def test_validate_finds_bad_d_and_dmin():
    M, K = 6, 1024
    W = synth.q4_k_weights(M, K, seed=19000).reshape(M, 4, 144)
    W[2, 3, 2:4] = np.array([0x7C00], dtype="<u2").view(np.uint8)   # dmin = +inf: super-block 11
    W[4, 1, 0:2] = np.array([0xFE00], dtype="<u2").view(np.uint8)   # d = NaN: super-block 17
    W[5, 0, 4:16] = 0xFF                                             # fields all ones: valid
    Wf = W.reshape(M, -1)
    assert gq.validate(Q4K, dev(Wf), K) == (2, 11)
    assert oracle.get().validate(Q4K, Wf, M, K) == (2, 11)


def test_shape_errors():
    L = gq._lib
    assert L.gq_type_nbytes(Q4K, 3, 4096) == 3 * 16 * 144
    assert L.gq_type_nbytes(Q4K, 3, 4096 + 32) == 0
    W = torch.zeros(144 * 4, dtype=torch.uint8, device="cuda")
    out = torch.empty(4 * 288, device="cuda")
    assert L.gq_dequant(Q4K, W.data_ptr(), 4, 288, out.data_ptr(), None) == gq.GQ_ERR_SHAPE
    assert "multiple of 256" in gq.gq_last_error()
    X = torch.zeros(1, 288, device="cuda")
    Y = torch.empty(1, 4, device="cuda")
    assert L.gq_mul_mat(Q4K, W.data_ptr(), 4, 288, X.data_ptr(), 1, Y.data_ptr(), None) == gq.GQ_ERR_SHAPE
    r = torch.empty(2, dtype=torch.int64, device="cuda")
    assert L.gq_validate(Q4K, W.data_ptr(), 4, 288, r.data_ptr(), None) == gq.GQ_ERR_SHAPE
