"""CUDA path against the CPU oracle, element by element, through the C ABI.

Dequantisation must be bit-exact (NaN == NaN); MUL_MAT must satisfy
|y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-5 for every element, with y_ref and
the sum from the fp64 oracle.  Inputs come from synth.py (seeded).
"""
import numpy as np
import pytest

import oracle
import synth
from golden_io import read_blocks, same_f32_bits
from gpu_util import assert_mul_mat_close, oracle_mul_mat

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import quantized_block_q4_gb300 as gq
else:  # collected on CPU machines, never run there (marked gpu)
    gq = None


def dev(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ------------------------------------------------------------------ dequant
DEQUANT_SHAPES = [(256, 1024), (11008, 4096), (4096, 11008), (4096, 4096), (32000, 4096), (14336, 4096),
                  (1, 32), (3, 64), (7, 288), (129, 256), (5, 8192)]


@pytest.mark.parametrize("M,K", DEQUANT_SHAPES)
def test_dequant_bit_exact(M, K):
    W = synth.q4_0_weights(M, K, seed=synth.seed_for(1, 0) + M + K)
    ref = oracle.get().dequant(W, M, K)
    out = gq.dequant_q4_0(dev(W), K)
    torch.cuda.synchronize()
    assert same_f32_bits(out.cpu().numpy(), ref).all()


def test_dequant_golden_blocks_and_signs():
    recs = read_blocks()
    W = np.concatenate([raw for _, raw, _ in recs])          # one row of len(recs) blocks
    K = 32 * len(recs)
    out = gq.dequant_q4_0(dev(W), K).cpu().numpy()[0]
    expect = np.concatenate([v for _, _, v in recs])
    assert same_f32_bits(out, expect).all()
    assert same_f32_bits(out, oracle.get().dequant(W, 1, K)[0]).all()


@pytest.mark.parametrize("offset", [1, 2, 6])
def test_dequant_unaligned(offset):
    M, K = 37, 288
    W = synth.q4_0_weights(M, K, seed=77)
    buf = torch.zeros(W.size + 64, dtype=torch.uint8, device="cuda")
    buf[offset:offset + W.size] = dev(W.reshape(-1))
    out = torch.full((M * K + 1,), float("nan"), dtype=torch.float32, device="cuda")
    gq.gq_dequant_q4_0(buf.data_ptr() + offset, M, K, out.data_ptr() + 4, None)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.isnan(got[0])
    assert same_f32_bits(got[1:].reshape(M, K), oracle.get().dequant(W, M, K)).all()


def test_dequant_scale_specials():
    # every scale class: +-0, subnormal, normal, max, +-inf, NaN; all codes 0..15
    d_bits = np.array([0x0000, 0x8000, 0x0001, 0x83FF, 0x3C00, 0xB555, 0x7BFF, 0x7C00, 0xFC00, 0x7E01],
                      dtype=np.uint16)
    nb = d_bits.size
    ramp = np.array([j | ((15 - j) << 4) for j in range(16)], dtype=np.uint8)  # every code, both nibbles
    qs = np.tile(ramp, (1, nb, 1))
    W = synth.blocks_from_parts(d_bits.reshape(1, nb), qs)
    out = gq.dequant_q4_0(dev(W), 32 * nb).cpu().numpy()
    assert same_f32_bits(out, oracle.get().dequant(W, 1, 32 * nb)).all()


def test_dequant_empty_and_errors():
    out = torch.empty(0, dtype=torch.float32, device="cuda")
    gq.gq_dequant_q4_0(torch.empty(0, dtype=torch.uint8, device="cuda"), 0, 64, out)
    with pytest.raises(gq.GQError) as e:
        gq.gq_dequant_q4_0(torch.empty(18, dtype=torch.uint8, device="cuda"), 1, 33, out)
    assert e.value.status == gq.GQ_ERR_SHAPE


# ------------------------------------------------------------------ mul_mat
def run_mm(W, X, M, K):
    Wd, Xd = dev(W), dev(X)
    Y = gq.mul_mat_q4_0(Wd, Xd)
    torch.cuda.synchronize()
    gq.gq_sync_status()
    return Y.cpu().numpy()


def check_mm(M, K, N, seed, label=""):
    W = synth.q4_0_weights(M, K, seed=seed)
    X = synth.activations(N, K, seed=seed + 1)
    y = run_mm(W, X, M, K)
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    return assert_mul_mat_close(y, y_ref, s_ref, label or f"M={M} K={K} N={N}")


def test_tiny_matvec():  # 256 x 1024, N = 1
    check_mm(256, 1024, 1, synth.seed_for(1, 0))


@pytest.mark.parametrize("M,K", [(11008, 4096), (4096, 11008)])
def test_ffn_decode(M, K):
    check_mm(M, K, 1, synth.seed_for(2, 0) + M)


@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("M", [4096, 32000])
def test_small_batch_decode(M, N):
    check_mm(M, 4096, N, synth.seed_for(3, N) + M)


@pytest.mark.parametrize("N", [1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 32, 33, 48, 63, 64, 65, 127, 128, 129, 200])
def test_n_edges(N):
    check_mm(129, 512, N, 900 + N)


@pytest.mark.parametrize("M", [1, 3, 15, 16, 17, 100, 255, 257])
@pytest.mark.parametrize("N", [1, 5, 64, 130])
def test_m_edges(M, N):
    check_mm(M, 768, N, 1000 + M * 7 + N)


@pytest.mark.parametrize("K", [32, 64, 96, 288, 1000 // 32 * 32, 2048 + 32])
@pytest.mark.parametrize("N", [1, 3, 70])
def test_k_not_multiple_of_256(K, N):
    check_mm(33, K, N, 2000 + K + N)


@pytest.mark.parametrize("K", [256, 512, 2304, 8448, 12288, 16384])
@pytest.mark.parametrize("N", [1, 16, 40, 64, 256])
def test_k_sweep(K, N):
    check_mm(80, K, N, 3000 + K + N)


def test_zero_k_writes_zeros():
    Y = torch.full((3, 5), 7.0, device="cuda")
    gq.gq_mul_mat_q4_0(torch.empty(0, dtype=torch.uint8, device="cuda"), 5, 0,
                       torch.empty(3, 0, device="cuda"), 3, Y)
    torch.cuda.synchronize()
    assert (Y.cpu().numpy() == 0).all()


def test_generic_path_matches():
    gq.gq_set_option(gq.GQ_OPT_FORCE_GENERIC, 1)
    try:
        check_mm(70, 1024, 5, 4001, "forced generic")
        check_mm(70, 1024, 80, 4002, "forced generic")
    finally:
        gq.gq_set_option(gq.GQ_OPT_FORCE_GENERIC, 0)


def test_unaligned_pointers_take_generic_path():
    M, K, N = 40, 512, 3
    W = synth.q4_0_weights(M, K, seed=4100)
    X = synth.activations(N, K, seed=4101)
    wbuf = torch.zeros(W.size + 32, dtype=torch.uint8, device="cuda")
    wbuf[3:3 + W.size] = dev(W.reshape(-1))
    xbuf = torch.zeros(N * K + 1, dtype=torch.float32, device="cuda")
    xbuf[1:] = dev(X.reshape(-1))
    Y = torch.zeros(N * M + 1, dtype=torch.float32, device="cuda")
    gq.gq_mul_mat_q4_0(wbuf.data_ptr() + 3, M, K, xbuf.data_ptr() + 4, N, Y.data_ptr() + 4)
    torch.cuda.synchronize()
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    assert_mul_mat_close(Y.cpu().numpy()[1:].reshape(N, M), y_ref, s_ref, "unaligned")


def test_output_guard_bytes_untouched():
    M, K = 100, 1024
    for N in (1, 8, 64, 100):
        W = synth.q4_0_weights(M, K, seed=4200 + N)
        X = synth.activations(N, K, seed=4300 + N)
        guard = 1024
        buf = torch.full((guard + N * M + guard,), -12345.0, dtype=torch.float32, device="cuda")
        Y = buf[guard:guard + N * M]
        gq.gq_mul_mat_q4_0(dev(W), M, K, dev(X), N, Y)
        torch.cuda.synchronize()
        b = buf.cpu().numpy()
        assert (b[:guard] == -12345.0).all() and (b[-guard:] == -12345.0).all()
        y_ref, s_ref = oracle_mul_mat(W, M, K, X)
        assert_mul_mat_close(b[guard:guard + N * M].reshape(N, M), y_ref, s_ref, f"guard N={N}")


def test_repeated_calls_are_deterministic():
    M, K, N = 300, 4096, 4
    W, X = dev(synth.q4_0_weights(M, K, seed=5)), dev(synth.activations(N, K, seed=6))
    a = gq.mul_mat_q4_0(W, X)
    b = gq.mul_mat_q4_0(W, X)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_shape_errors():
    W = torch.zeros(18, dtype=torch.uint8, device="cuda")
    X = torch.zeros(1, 32, device="cuda")
    Y = torch.zeros(1, 1, device="cuda")
    with pytest.raises(gq.GQError) as e:
        gq.gq_mul_mat_q4_0(W, 1, 33, X, 1, Y)
    assert e.value.status == gq.GQ_ERR_SHAPE
    with pytest.raises(gq.GQError) as e:
        gq.gq_mul_mat_q4_0(W, -1, 32, X, 1, Y)
    assert e.value.status == gq.GQ_ERR_SHAPE
    with pytest.raises(gq.GQError) as e:
        gq.gq_mul_mat_q4_0(0, 1, 32, X, 1, Y)
    assert e.value.status == gq.GQ_ERR_NULL


def test_nonfinite_scale_propagates():
    M, K, N = 16, 256, 2
    W = synth.q4_0_weights(M, K, seed=8)
    Wv = W.reshape(M, K // 32, 18)
    Wv[3, 2, 0:2] = np.frombuffer(np.uint16(0x7C00).tobytes(), np.uint8)  # +inf scale
    X = synth.activations(N, K, seed=9)
    y = run_mm(W, X, M, K)
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    assert (np.isnan(y_ref[:, 3]) | np.isinf(y_ref[:, 3])).all()
    assert (np.isnan(y[:, 3]) | np.isinf(y[:, 3])).all()
    rest = [m for m in range(M) if m != 3]
    assert_mul_mat_close(y[:, rest], y_ref[:, rest], s_ref[:, rest], "finite rows")


# ------------------------------------------------------------------ prefill (tensor cores)
def sampled_rows(M, count, seed):
    rng = np.random.Generator(np.random.SFC64(seed))
    rows = np.concatenate([np.arange(min(128, M)), np.arange(max(0, M - 128), M),
                           rng.integers(0, M, count)])
    return np.unique(rows)


def test_prefill_full_size_sampled_rows():
    """14336 x 4096 weights, 512 tokens (the prefill workload): every column of
    a seeded sample of rows (first and last tile included) against the oracle."""
    M, K, N = 14336, 4096, 512
    W = synth.q4_0_weights(M, K, seed=synth.seed_for(4, 0))
    X = synth.activations(N, K, seed=synth.seed_for(4, 1))
    y = run_mm(W, X, M, K)
    rows = sampled_rows(M, 256, 41)
    y_ref, s_ref = oracle_mul_mat(W.reshape(M, -1)[rows], len(rows), K, X)
    assert_mul_mat_close(y[:, rows], y_ref, s_ref, "prefill sampled rows")


@pytest.mark.parametrize("N", [64, 96, 128, 129, 256, 300, 512, 513])
def test_prefill_n_tiles(N):
    check_mm(384, 1024, N, 5000 + N)


@pytest.mark.parametrize("M,K,N", [(256, 1024, 2048), (130, 512, 4099)])
def test_prefill_many_token_tiles(M, K, N):
    """Long batches: 8 and 17 token tiles of 256 (the last one ragged) per row tile."""
    check_mm(M, K, N, 5100 + N)


@pytest.mark.parametrize("opt,val", [("GQ_OPT_PREFILL_PAIR", 1), ("GQ_OPT_PREFILL_TILE_N", 128)])
@pytest.mark.parametrize("M,N", [(384, 129), (384, 300), (640, 513), (130, 257)])
def test_prefill_kernel_options(opt, val, M, N):
    """The 2-SM (CTA pair) kernel and the 128-wide tile variant, each against the oracle."""
    code = getattr(gq, opt)
    old = gq.gq_get_option(code)
    gq.gq_set_option(code, val)
    try:
        check_mm(M, 1024, N, 5100 + M + N)
    finally:
        gq.gq_set_option(code, old)


def _with_option(code, val, fn):
    old = gq.gq_get_option(code)
    gq.gq_set_option(code, val)
    try:
        return fn()
    finally:
        gq.gq_set_option(code, old)


# Every tile split along k into n pieces (partial sums through the workspace,
# summed in k order by whichever piece arrives last).  T = ceil(M/128) *
# ceil(N/BN) tiles of K/256 chunks; n is capped at the chunk count.
#   384x1024 (4 chunks), N=300: 2, 3, 4 and 7 (-> 4) pieces; N=100: the 128-wide tile;
#   640x2048 (8 chunks), N=513: 3 and 8 pieces; 130 rows: ragged last row block;
#   N = 16, 17, 40: a 128-wide tile with 16, 17 or 40 valid columns (only those
#   are published and reduced).
@pytest.mark.parametrize("M,K,N,n", [(384, 1024, 300, 2), (384, 1024, 300, 3), (384, 1024, 300, 4),
                                     (384, 1024, 300, 7), (384, 1024, 100, 2), (640, 2048, 513, 3),
                                     (640, 2048, 513, 8), (130, 1024, 257, 3), (384, 1024, 16, 4),
                                     (384, 1024, 17, 3), (640, 2048, 40, 2)])
def test_prefill_split_every_tile(M, K, N, n):
    _with_option(gq.GQ_OPT_PREFILL_STREAMK, n, lambda: check_mm(M, K, N, 5200 + M + N + n, f"k-split n={n}"))


# The default planner on a GPU of `slots` SMs: 640x8192, N=513 is 15 tiles of
# 32 chunks.  4 slots: 3-4 whole tiles per CTA; 6: 2 whole tiles each and the
# last 3 tiles in 2 pieces; 7: 2 whole tiles each and the last tile in 7
# pieces; 40: no whole tiles, every tile in 2 pieces; 16: one tile per CTA.
@pytest.mark.parametrize("slots", [4, 6, 7, 16, 40])
def test_prefill_schedule(slots):
    _with_option(gq.GQ_OPT_PREFILL_SLOTS, slots,
                 lambda: check_mm(640, 8192, 513, 5300 + slots, f"schedule on {slots} SMs"))


# CTA pairs (256-row tiles): 640x2048, N=513 is 3 x 3 pair tiles of 8 chunks;
# 130 rows: the second CTA of each pair has no rows.
@pytest.mark.parametrize("M,K,N,n,slots", [(640, 2048, 513, 3, 0), (640, 2048, 513, 8, 0), (384, 1024, 300, 2, 0),
                                           (130, 1024, 300, 3, 0), (640, 8192, 513, 1, 2), (640, 8192, 513, 1, 4),
                                           (640, 8192, 513, 0, 4)])
def test_prefill_pair_split_and_schedule(M, K, N, n, slots):
    def run():
        return _with_option(gq.GQ_OPT_PREFILL_STREAMK, n, lambda: _with_option(
            gq.GQ_OPT_PREFILL_SLOTS, slots, lambda: check_mm(M, K, N, 5500 + M + N + n + slots, "pair")))
    _with_option(gq.GQ_OPT_PREFILL_PAIR, 1, run)


def test_prefill_split_is_deterministic():
    """Split tiles are summed in k order, so repeated calls agree bit for bit."""
    M, K, N = 640, 2048, 513
    W = dev(synth.q4_0_weights(M, K, seed=5300))
    X = dev(synth.activations(N, K, seed=5301))

    def run():
        ys = [gq.mul_mat_q4_0(W, X) for _ in range(4)]
        torch.cuda.synchronize()
        return ys
    ys = _with_option(gq.GQ_OPT_PREFILL_STREAMK, 3, run)
    for y in ys[1:]:
        assert torch.equal(ys[0], y)


def test_prefill_whole_tiles_only_matches_oracle():
    _with_option(gq.GQ_OPT_PREFILL_STREAMK, 0, lambda: check_mm(640, 2048, 513, 5400, "whole tiles"))


@pytest.mark.parametrize("tile_n", [0, 128, 256])
@pytest.mark.parametrize("M,K", [(4096, 4096), (4096, 11008), (11008, 4096)])
def test_prefill_full_size_split_sampled_rows(M, K, tile_n):
    """The sweep's N = 512 shapes under the planner's own choice (tile_n = 0:
    4096 x 4096 in 128-token tiles, 11008 x 4096 in two waves of whole tiles,
    4096 x 11008 split in two along k) and with each tile width forced (at 256
    tokens 4096 x 4096 has 64 tiles, which the planner may split along k).
    Sampled rows against the oracle."""
    N = 512
    W = synth.q4_0_weights(M, K, seed=synth.seed_for(5, M + K))
    X = synth.activations(N, K, seed=synth.seed_for(5, M + K + 1))
    y = _with_option(gq.GQ_OPT_PREFILL_TILE_N, tile_n, lambda: run_mm(W, X, M, K))
    rows = sampled_rows(M, 128, 43)
    y_ref, s_ref = oracle_mul_mat(W.reshape(M, -1)[rows], len(rows), K, X)
    assert_mul_mat_close(y[:, rows], y_ref, s_ref, f"{M}x{K} tile_n={tile_n}")


@pytest.mark.parametrize("M,K,N", [(4096, 4096, 16), (4096, 11008, 24), (32000, 4096, 16)])
def test_prefill_small_batch_full_size_sampled_rows(M, K, N):
    """The small-batch shapes on the tensor-core kernel under the planner's
    choice (4096 x 4096 at 16 tokens: 32 tiles split in 4 along k; 32000 x
    4096: two waves of whole tiles).  Sampled rows against the oracle."""
    W = synth.q4_0_weights(M, K, seed=synth.seed_for(3, M + K + N))
    X = synth.activations(N, K, seed=synth.seed_for(3, M + K + N + 1))
    y = run_mm(W, X, M, K)
    rows = sampled_rows(M, 128, 47)
    y_ref, s_ref = oracle_mul_mat(W.reshape(M, -1)[rows], len(rows), K, X)
    assert_mul_mat_close(y[:, rows], y_ref, s_ref, f"{M}x{K} N={N}")


def test_f32_to_bf16_matches_torch_rounding():
    x = torch.from_numpy(synth.activations(7, 1000, seed=12)).cuda().reshape(-1)
    x[:6] = torch.tensor([float("nan"), float("inf"), -float("inf"), 0.0, -0.0, 1e-40], device="cuda")
    y = torch.empty(x.numel(), dtype=torch.int16, device="cuda")
    gq.gq_f32_to_bf16(x, y, x.numel())
    ref = x.to(torch.bfloat16).view(torch.int16)
    torch.cuda.synchronize()
    nan = torch.isnan(x)
    assert torch.equal(y[~nan], ref[~nan])
    assert torch.isnan(y.view(torch.bfloat16)[nan].float()).all()


@pytest.mark.parametrize("N", [1, 7, 16, 64, 200])
def test_bf16_activation_entry(N):
    M, K = 257, 2048
    W = synth.q4_0_weights(M, K, seed=6000 + N)
    X = synth.activations(N, K, seed=6100 + N)
    xb = torch.from_numpy(X).cuda().to(torch.bfloat16)
    Y = torch.empty(N, M, device="cuda")
    gq.gq_mul_mat_q4_0_bf16x(dev(W), M, K, xb.view(torch.int16), N, Y)
    torch.cuda.synchronize()
    gq.gq_sync_status()
    y_ref, s_ref = oracle_mul_mat(W, M, K, xb.float().cpu().numpy())
    assert_mul_mat_close(Y.cpu().numpy(), y_ref, s_ref, f"bf16x N={N}")


def test_prefill_threshold_option_switches_kernels():
    M, K, N = 200, 1024, 12
    W = synth.q4_0_weights(M, K, seed=7000)
    X = synth.activations(N, K, seed=7001)
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    old = gq.gq_get_option(gq.GQ_OPT_PREFILL_MIN_N)
    try:
        gq.gq_set_option(gq.GQ_OPT_PREFILL_MIN_N, 1)           # tensor-core path for N = 20
        a = run_mm(W, X, M, K)
    finally:
        gq.gq_set_option(gq.GQ_OPT_PREFILL_MIN_N, old)
    b = run_mm(W, X, M, K)                                      # decode path
    assert_mul_mat_close(a, y_ref, s_ref, "tensor-core path")
    assert_mul_mat_close(b, y_ref, s_ref, "decode path")


def test_prefill_dequant_is_single_rounded_bf16():
    """One-hot activation rows: every output is one weight times 1, so the
    tensor-core path must return exactly RN_bf16(d*(q-8)) (torch's bf16
    rounding of the oracle's fp32 dequant)."""
    M, K, N = 300, 1024, 96
    W = synth.q4_0_weights(M, K, seed=7100)
    ks = np.random.Generator(np.random.SFC64(7101)).integers(0, K, N)
    X = np.zeros((N, K), dtype=np.float32)
    X[np.arange(N), ks] = 1.0
    xb = torch.from_numpy(X).cuda().to(torch.bfloat16)
    Y = torch.empty(N, M, device="cuda")
    gq.gq_mul_mat_q4_0_bf16x(dev(W), M, K, xb.view(torch.int16), N, Y)
    torch.cuda.synchronize()
    w_bf16 = torch.from_numpy(oracle.get().dequant(W, M, K)).to(torch.bfloat16).float().numpy()
    expect = w_bf16[:, ks].T                                  # [N, M]
    assert same_f32_bits(np.abs(Y.cpu().numpy()), np.abs(expect)).all()


def test_weights_static_option_gives_identical_results():
    M, K, N = 2000, 4096, 3
    W = dev(synth.q4_0_weights(M, K, seed=7200))
    X = dev(synth.activations(N, K, seed=7201))
    a = gq.mul_mat_q4_0(W, X)
    gq.gq_set_option(gq.GQ_OPT_WEIGHTS_STATIC, 1)
    try:
        b = gq.mul_mat_q4_0(W, X)
        c = gq.mul_mat_q4_0(W, X)
    finally:
        gq.gq_set_option(gq.GQ_OPT_WEIGHTS_STATIC, 0)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(b, c)


def test_back_to_back_dependent_calls():
    """Each call's X is the previous call's Y: programmatic dependent launch
    must still order the reads after the producer kernel."""
    K = 4096
    Ws = [synth.q4_0_weights(K, K, seed=7300 + i) for i in range(4)]
    x0 = synth.activations(2, K, seed=7310)
    xs = [dev(x0)]
    for W in Ws:
        xs.append(gq.mul_mat_q4_0(dev(W), xs[-1]))
    torch.cuda.synchronize()
    x = x0
    for i, W in enumerate(Ws):
        y_ref, s_ref = oracle_mul_mat(W, K, K, x)
        got = xs[i + 1].cpu().numpy()
        assert_mul_mat_close(got, y_ref, s_ref, f"chain step {i}")
        x = got.astype(np.float32)      # continue from what the GPU produced


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("M,K,N", [(4096, 4096, 1), (300, 11008, 3), (33, 2304, 8), (1000, 4096, 12),
                                   (530, 8192, 16)])
def test_decode_variants(variant, M, K, N):
    old = gq.gq_get_option(gq.GQ_OPT_DECODE_VARIANT)
    gq.gq_set_option(gq.GQ_OPT_DECODE_VARIANT, variant)
    try:
        _with_option(gq.GQ_OPT_PREFILL_MIN_N, 65, lambda: check_mm(M, K, N, 7400 + M + N, f"variant {variant}"))
    finally:
        gq.gq_set_option(gq.GQ_OPT_DECODE_VARIANT, old)


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
@pytest.mark.parametrize("M,K,N", [(700, 4096, 24), (260, 8192, 32)])
def test_decode_variants_17_to_32_tokens(variant, M, K, N):
    """17..32 tokens on the decode kernel (the tensor-core threshold raised):
    four n8 token tiles, one or several x chunks."""
    def run():
        return _with_option(gq.GQ_OPT_PREFILL_MIN_N, 65, lambda: check_mm(M, K, N, 7450 + M + N, f"variant {variant}"))
    _with_option(gq.GQ_OPT_DECODE_VARIANT, variant, run)


@pytest.mark.parametrize("weights_static", [0, 1])
def test_prefill_back_to_back_dependent_calls(weights_static):
    """Tensor-core calls launched with programmatic dependent launch, each X
    the previous call's Y: the conversion and the MUL_MAT must wait for the
    kernel that produced their input (with WEIGHTS_STATIC only W streams
    early)."""
    K, N = 2048, 64
    Ws = [synth.q4_0_weights(K, K, seed=7500 + i) for i in range(4)]
    x0 = synth.activations(N, K, seed=7510)

    def run():
        xs = [dev(x0)]
        for W in Ws:
            xs.append(gq.mul_mat_q4_0(dev(W), xs[-1]))
        torch.cuda.synchronize()
        gq.gq_sync_status()
        return xs
    xs = _with_option(gq.GQ_OPT_WEIGHTS_STATIC, weights_static, run)
    x = x0
    for i, W in enumerate(Ws):
        y_ref, s_ref = oracle_mul_mat(W, K, K, x)
        got = xs[i + 1].cpu().numpy()
        assert_mul_mat_close(got, y_ref, s_ref, f"prefill chain step {i}")
        x = got.astype(np.float32)


def test_prefill_quantize_then_mul_mat():
    """W written on the device by the quantizer right before the tensor-core
    MUL_MAT that reads it (WEIGHTS_STATIC off: W is read after the wait)."""
    M, K, N = 900, 2048, 80
    Wf = synth.activations(M, K, seed=7520)
    X = synth.activations(N, K, seed=7521)
    Wq = torch.empty(gq.gq_q4_0_nbytes(M, K), dtype=torch.uint8, device="cuda")
    Wfd, Xd = dev(Wf), dev(X)
    Y = torch.empty(N, M, device="cuda")
    for _ in range(2):
        gq.gq_quantize_q4_0(Wfd, M, K, Wq)
        gq.gq_mul_mat_q4_0(Wq, M, K, Xd, N, Y)
        Wfd.mul_(-1.0)  # the next round quantizes other values into the same W buffer
    torch.cuda.synchronize()
    gq.gq_sync_status()
    Wq_ref = oracle.get().quantize(-Wf)  # the second round quantized the negated values
    assert np.array_equal(Wq.cpu().numpy().reshape(Wq_ref.shape), Wq_ref)
    y_ref, s_ref = oracle_mul_mat(Wq_ref, M, K, X)
    assert_mul_mat_close(Y.cpu().numpy(), y_ref, s_ref, "quantize -> mul_mat")


@pytest.mark.parametrize("streamk", [1, 3])
def test_prefill_same_output_and_scratch_back_to_back(streamk):
    """Consecutive tensor-core calls into one Y (and, split along k, through
    reused scratch): the last call's result must be what remains."""
    M, K, N = 640, 2048, 300
    Ws = [synth.q4_0_weights(M, K, seed=7530 + i) for i in range(3)]
    X = synth.activations(N, K, seed=7535)
    Wd, Xd = [dev(w) for w in Ws], dev(X)
    Y = torch.empty(N, M, device="cuda")
    Ylast = torch.empty(N, M, device="cuda")

    def run():
        for _ in range(3):
            for w in Wd:
                gq.gq_mul_mat_q4_0(w, M, K, Xd, N, Y)
            gq.gq_mul_mat_q4_0(Wd[1], M, K, Xd, N, Ylast)
        torch.cuda.synchronize()
        gq.gq_sync_status()
    _with_option(gq.GQ_OPT_PREFILL_STREAMK, streamk, run)
    y_ref, s_ref = oracle_mul_mat(Ws[2], M, K, X)
    assert_mul_mat_close(Y.cpu().numpy(), y_ref, s_ref, "last writer wins")
    y_ref, s_ref = oracle_mul_mat(Ws[1], M, K, X)
    assert_mul_mat_close(Ylast.cpu().numpy(), y_ref, s_ref, "interleaved call")


@pytest.mark.parametrize("N", [2, 3, 4])
@pytest.mark.parametrize("M,K", [(4096, 4096), (1000, 2048), (4096, 11008)])
def test_small_batch_co_resident_cta(M, K, N):
    """2-4 tokens under both promises on matrices of at most one 32-row tile
    per SM: the 4-warp CTA (two launches share an SM), back to back."""
    Ws = [synth.q4_0_weights(M, K, seed=8100 + i + N) for i in range(2)]
    Xs = [synth.activations(N, K, seed=8110 + i + N) for i in range(2)]
    Wd, Xd = [dev(w) for w in Ws], [dev(x) for x in Xs]
    Ys = [torch.empty(N, M, device="cuda") for _ in range(2)]

    def run():
        for _ in range(3):
            for w, x, y in zip(Wd, Xd, Ys):
                gq.gq_mul_mat_q4_0(w, M, K, x, N, y)
        torch.cuda.synchronize()
        gq.gq_sync_status()
    _with_option(gq.GQ_OPT_X_STATIC, 1, lambda: _with_option(gq.GQ_OPT_WEIGHTS_STATIC, 1, run))
    for i in range(2):
        y_ref, s_ref = oracle_mul_mat(Ws[i], M, K, Xs[i])
        assert_mul_mat_close(Ys[i].cpu().numpy(), y_ref, s_ref, f"{N} tokens, call {i}")


@pytest.mark.parametrize("M,K", [(4096, 4096), (11008, 4096), (4096, 11008)])
def test_x_static_back_to_back_independent_calls(M, K):
    """X_STATIC + WEIGHTS_STATIC: calls whose X no preceding kernel writes may
    read X and compute before that kernel finishes; Y is written after it.
    Several calls in a row, each checked against the oracle."""
    Ws = [synth.q4_0_weights(M, K, seed=7800 + i) for i in range(3)]
    Xs = [synth.activations(1, K, seed=7810 + i) for i in range(3)]
    Wd, Xd = [dev(w) for w in Ws], [dev(x) for x in Xs]
    Ys = [torch.empty(1, M, device="cuda") for _ in range(3)]

    def run():
        for _ in range(3):  # repeated: the later rounds overwrite Y while earlier calls may still run
            for w, x, y in zip(Wd, Xd, Ys):
                gq.gq_mul_mat_q4_0(w, M, K, x, 1, y)
        torch.cuda.synchronize()
        gq.gq_sync_status()
    _with_option(gq.GQ_OPT_X_STATIC, 1, lambda: _with_option(gq.GQ_OPT_WEIGHTS_STATIC, 1, run))
    for i in range(3):
        y_ref, s_ref = oracle_mul_mat(Ws[i], M, K, Xs[i])
        assert_mul_mat_close(Ys[i].cpu().numpy(), y_ref, s_ref, f"x-static call {i}")


def _chain_rounds(project, make_x, rounds=4):
    """A writer kernel produces X, then three projections of it: the first
    call without GQ_OPT_X_STATIC, the next two with it (the pattern the
    promise allows).  Each round writes another X, so a projection that read
    X before its writer finished would carry the previous round's values.
    Returns the last round's X (host) and three outputs."""
    out = None
    for r in range(rounds):
        x = make_x(r)
        ys = []
        for i in range(3):
            gq.gq_set_option(gq.GQ_OPT_X_STATIC, 0 if i == 0 else 1)
            ys.append(project(i, x))
        gq.gq_set_option(gq.GQ_OPT_X_STATIC, 0)
        out = (x, ys)
    torch.cuda.synchronize()
    gq.gq_sync_status()
    return out


def test_x_static_chain_after_a_writer_decode():
    """Decode: X of the projections is the Y of the MUL_MAT right before them."""
    M0 = K = 4096
    W0 = synth.q4_0_weights(M0, 2048, seed=7900)
    Ws = [synth.q4_0_weights(4096, K, seed=7901 + i) for i in range(3)]
    W0d, Wd = dev(W0), [dev(w) for w in Ws]
    X0s = [dev(synth.activations(1, 2048, seed=7910 + r)) for r in range(4)]
    Y1 = torch.empty(1, K, device="cuda")
    Ys = [torch.empty(1, 4096, device="cuda") for _ in range(3)]

    def make_x(r):
        gq.gq_mul_mat_q4_0(W0d, M0, 2048, X0s[r], 1, Y1)  # the writer of X (no promise)
        return Y1

    def project(i, x):
        gq.gq_mul_mat_q4_0(Wd[i], 4096, K, x, 1, Ys[i])
        return Ys[i]
    old = gq.gq_get_option(gq.GQ_OPT_X_STATIC)
    try:
        x, ys = _with_option(gq.GQ_OPT_WEIGHTS_STATIC, 1, lambda: _chain_rounds(project, make_x))
    finally:
        gq.gq_set_option(gq.GQ_OPT_X_STATIC, old)
    xh = x.cpu().numpy()
    for i in range(3):
        y_ref, s_ref = oracle_mul_mat(Ws[i], 4096, K, xh)
        assert_mul_mat_close(ys[i].cpu().numpy(), y_ref, s_ref, f"decode projection {i} of the last round")


@pytest.mark.parametrize("M,K,N", [(4096, 4096, 512), (11008, 4096, 300), (640, 2048, 64), (4096, 4096, 16),
                                   (4096, 11008, 512)])
def test_x_static_chain_after_a_writer_tensor_core(M, K, N):
    """gq_mul_mat_q4_0_bf16x: X_bf16 is written by the activation conversion
    right before the first projection; the other two carry the promise and
    may start their MMAs while the kernels ahead of them finish (and run whole
    256-token tiles, or whole 128-token tiles at 16 tokens, where the first
    call's plan splits them along k)."""
    Ws = [synth.q4_0_weights(M, K, seed=7920 + i) for i in range(3)]
    Wd = [dev(w) for w in Ws]
    Xfs = [dev(synth.activations(N, K, seed=7930 + r)) for r in range(4)]
    Xb = torch.empty(N, K, dtype=torch.int16, device="cuda")
    Ys = [torch.empty(N, M, device="cuda") for _ in range(3)]

    def make_x(r):
        gq.gq_f32_to_bf16(Xfs[r], Xb, N * K)  # the writer of X
        return Xb

    def project(i, x):
        gq.gq_mul_mat_q4_0_bf16x(Wd[i], M, K, x, N, Ys[i])
        return Ys[i]
    old = gq.gq_get_option(gq.GQ_OPT_X_STATIC)
    try:
        x, ys = _with_option(gq.GQ_OPT_WEIGHTS_STATIC, 1, lambda: _chain_rounds(project, make_x))
    finally:
        gq.gq_set_option(gq.GQ_OPT_X_STATIC, old)
    xh = (x.cpu().numpy().astype(np.int32).astype(np.uint32) << 16).view(np.float32)  # bf16 bits -> fp32
    rows = sampled_rows(M, 96, 79)
    for i in range(3):
        y_ref, s_ref = oracle_mul_mat(Ws[i].reshape(M, -1)[rows], len(rows), K, xh)
        assert_mul_mat_close(ys[i].cpu().numpy()[:, rows], y_ref, s_ref, f"tensor-core projection {i}")


@pytest.mark.parametrize("stages", [1, 2, 3, 8])
def test_decode_early_stages_option(stages):
    def run():
        return _with_option(gq.GQ_OPT_WEIGHTS_STATIC, 1, lambda: check_mm(4096, 4096, 1, 7900 + stages, "early"))
    _with_option(gq.GQ_OPT_DECODE_EARLY_STAGES, stages, run)
