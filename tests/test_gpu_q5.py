"""Q5_0 and Q5_1 on the GPU against the oracle: dequantisation bit for bit,
MUL_MAT within |y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-5 (fp64 oracle) on
the mma.sync decode kernel (N < 16) and the tensor-core kernel (N >= 16), both
for K % 256 == 0 and aligned pointers, and the scalar kernel (other K,
unaligned, forced); validation of d (and Q5_1's m).  Inputs:
synth.typed_weights (fp16 d ~ U[0.0025, 0.01], Q5_1 m ~ U[-0.16, 0], random
high-bit and code bytes) and N(0, 1) activations."""
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

TYPES = [4, 5]  # GQ_TYPE_Q5_0, GQ_TYPE_Q5_1 (same numbering as oracle.TYPE_*)
NAMES = {4: "q5_0", 5: "q5_1"}
BB = {4: 22, 5: 24}


def dev(a):
    return torch.from_numpy(np.array(a, copy=True)).cuda()


def _with_option(code, val, fn):
    old = gq.gq_get_option(code)
    gq.gq_set_option(code, val)
    try:
        return fn()
    finally:
        gq.gq_set_option(code, old)


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K", [(1, 32), (7, 96), (129, 288), (256, 1024), (11008, 4096), (4096, 11008)])
def test_dequant_bit_exact(qtype, M, K):
    W = synth.typed_weights(qtype, M, K, seed=19100 + M + K + qtype)
    got = gq.dequant(qtype, dev(W), K).cpu().numpy()
    assert same_f32_bits(got, oracle.get().dequant_typed(qtype, W, M, K)).all()


def test_dequant_golden_blocks():
    blocks = read_typed_blocks("q5_blocks.txt")
    assert blocks
    for tname, name, raw, values in blocks:
        qtype = {"q5_0": 4, "q5_1": 5}[tname]
        got = gq.dequant(qtype, dev(raw), 32).cpu().numpy()[0]
        assert same_f32_bits(got, values).all(), name


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
def test_dequant_unaligned(qtype):
    M, K = 37, 320
    W = synth.typed_weights(qtype, M, K, seed=19200 + qtype)
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
    gq.gq_sync_status()
    rows = np.arange(M) if sample is None else np.sort(np.random.default_rng(seed).choice(M, sample, replace=False))
    Wr = W.reshape(M, K // 32 * BB[qtype])[rows]
    y_ref, s_ref = oracle.get().mul_mat_typed(qtype, Wr, len(rows), K, X, nthreads=cores())
    return assert_mul_mat_close(y[:, rows], y_ref, s_ref, f"{NAMES[qtype]} M={M} K={K} N={N}")


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K,N", [(129, 96, 4), (77, 288, 5), (1, 32, 1), (64, 288, 40), (300, 800, 3)])
def test_scalar_kernel_matches_oracle(qtype, M, K, N):
    """K % 256 != 0: the scalar kernel (row-bulk copies for aligned rows of a
    multiple of 16 bytes, else plain loads)."""
    check(qtype, M, K, N, seed=19300 + M + K + N + qtype)


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K,N", [(256, 1024, 1), (300, 512, 3), (1000, 8192, 8), (33, 1024, 15), (500, 4096, 9),
                                   (700, 256, 1), (4096, 4096, 2)])
def test_decode_kernel_matches_oracle(qtype, M, K, N):
    """1-15 tokens with K % 256 == 0: the mma.sync decode kernel on 22- / 24-byte
    blocks (one and two token tiles, ragged rows, several x chunks)."""
    check(qtype, M, K, N, seed=19350 + M + K + N + qtype)


@pytest.mark.parametrize("static", [0, 1])
@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K", [(11008, 4096), (4096, 11008), (32000, 4096)])
def test_decode_sweep_shapes(qtype, M, K, static):
    """N = 1 on the sweep's shapes with and without the static promises (the
    co-resident 4-warp CTA and the 8-warp CTA)."""
    def run():
        return check(qtype, M, K, 1, seed=19370 + M + static + qtype, sample=96)
    _with_option(gq.GQ_OPT_WEIGHTS_STATIC, static, lambda: _with_option(gq.GQ_OPT_X_STATIC, static, run))


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("N,x_scale", [(1, 1e-6), (5, 1e-6), (1, 1e5), (12, 1e5)])
def test_decode_small_and_large_x(qtype, N, x_scale):
    """Activations far below 1 (1e-6 N(0,1), O(1) weights) and beyond fp16's
    range (1e5 N(0,1)): the decode kernel's power-of-two staging."""
    M, K = 600, 4096
    W = synth.typed_weights(qtype, M, K, seed=19380 + N + qtype, d_scale=100.0 if x_scale < 1 else 1.0)
    X = synth.activations(N, K, seed=19381 + N) * np.float32(x_scale)
    y = gq.mul_mat(qtype, dev(W), dev(X)).cpu().numpy()
    gq.gq_sync_status()
    y_ref, s_ref = oracle.get().mul_mat_typed(qtype, W, M, K, X, nthreads=cores())
    assert np.isfinite(y).all()
    assert_mul_mat_close(y, y_ref, s_ref, f"{NAMES[qtype]} x scale {x_scale} N={N}")


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K,N", [(300, 512, 16), (129, 1024, 100), (1000, 2048, 257), (64, 256, 128),
                                   (700, 4096, 64), (130, 768, 17)])
def test_tensor_core_path_matches_oracle(qtype, M, K, N):
    """N >= 16 with K % 256 == 0: the tcgen05 kernel with 176- or 192-byte raw
    rows (every dequant group's window position, several row tiles, ragged
    M and N, split and whole tiles)."""
    check(qtype, M, K, N, seed=19400 + M + N + qtype)


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K,N", [(11008, 4096, 1), (4096, 11008, 1), (14336, 4096, 512), (4096, 11008, 512)])
def test_full_size_sampled_rows(qtype, M, K, N):
    check(qtype, M, K, N, seed=19500 + N + qtype, sample=48)


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("N", [32, 4])
def test_fast_and_scalar_paths_agree(qtype, N):
    """N = 32 (tensor core) and N = 4 (decode kernel), each also through the
    scalar kernel (GQ_OPT_FORCE_GENERIC), all against the oracle."""
    M, K = 500, 1024
    check(qtype, M, K, N, seed=19600 + qtype + N)
    _with_option(gq.GQ_OPT_FORCE_GENERIC, 1, lambda: check(qtype, M, K, N, seed=19600 + qtype + N))


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
def test_mul_mat_unaligned(qtype):
    M, K, N = 40, 256, 3
    W = synth.typed_weights(qtype, M, K, seed=19700 + qtype)
    X = synth.activations(N, K, 19701)
    wb = torch.zeros(W.size + 8, dtype=torch.uint8, device="cuda")
    wb[1:1 + W.size] = dev(W.reshape(-1))
    xb = torch.zeros(N * K + 1, device="cuda")
    xb[1:] = dev(X).reshape(-1)
    Y = torch.empty(N, M, device="cuda")
    gq.gq_mul_mat(qtype, wb.data_ptr() + 1, M, K, xb.data_ptr() + 4, N, Y)
    torch.cuda.synchronize()
    gq.gq_sync_status()
    y_ref, s_ref = oracle.get().mul_mat_typed(qtype, W, M, K, X)
    assert_mul_mat_close(Y.cpu().numpy(), y_ref, s_ref, "unaligned")


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
def test_validate(qtype):
    M, K = 5, 256
    bb = BB[qtype]
    W = synth.typed_weights(qtype, M, K, seed=19800 + qtype).reshape(M, 8, bb)
    W[1, 5, 0:2] = np.array([0x7C00], dtype="<u2").view(np.uint8)   # d = inf: block 13
    W[3, 2, 2:4] = np.array([0xFE00], dtype="<u2").view(np.uint8)   # Q5_1: m = NaN (block 26); Q5_0: high bits
    Wf = W.reshape(M, -1)
    want = (2, 13) if qtype == 5 else (1, 13)
    assert gq.validate(qtype, dev(Wf), K) == want
    assert oracle.get().validate(qtype, Wf, M, K) == want


@pytest.mark.parametrize("qtype", [3, 4, 5], ids=["q4_k", "q5_0", "q5_1"])
def test_empty_sizes(qtype):
    """M, N == 0: nothing happens; K == 0: Y is zeros (the empty sum); validation
    of an empty matrix reports nothing."""
    L = gq._lib
    Y = torch.full((3, 5), float("nan"), device="cuda")
    X = torch.zeros(3, 256, device="cuda")
    W = torch.zeros(5 * gq.TYPE_BLOCK_BYTES[qtype] * (256 // gq.TYPE_BLOCK_WEIGHTS[qtype]), dtype=torch.uint8,
                    device="cuda")
    assert L.gq_mul_mat(qtype, W.data_ptr(), 0, 256, X.data_ptr(), 3, Y.data_ptr(), None) == gq.GQ_OK
    assert L.gq_mul_mat(qtype, W.data_ptr(), 5, 256, X.data_ptr(), 0, Y.data_ptr(), None) == gq.GQ_OK
    torch.cuda.synchronize()
    assert torch.isnan(Y).all()
    assert L.gq_mul_mat(qtype, W.data_ptr(), 5, 0, X.data_ptr(), 3, Y.data_ptr(), None) == gq.GQ_OK
    torch.cuda.synchronize()
    assert (Y == 0).all()
    out = torch.empty(1, device="cuda")
    assert L.gq_dequant(qtype, W.data_ptr(), 0, 256, out.data_ptr(), None) == gq.GQ_OK
    r = torch.full((2,), 7, dtype=torch.int64, device="cuda")
    assert L.gq_validate(qtype, W.data_ptr(), 0, 256, r.data_ptr(), None) == gq.GQ_OK
    torch.cuda.synchronize()
    assert r.cpu().tolist() == [0, -1]  # count 0, first = UINT64_MAX read as int64
    assert L.gq_type_nbytes(qtype, 0, 256) == 0
