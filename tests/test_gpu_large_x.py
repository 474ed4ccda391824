"""Activations beyond the fp16 range on the decode kernel, against the oracle.

The decode kernel stages x as fp16 (largest finite value 65504).  Tokens whose
x reaches 2^15 in a warp's blocks are staged scaled by an exact power of two
and their partial sums scaled back; every element must still satisfy
|y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-5 (fp64 oracle).  Inputs:
synth.wide_range_activations (N(0, 1) with a quarter of some tokens' blocks
scaled by 1e5 .. 1e9, or more).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_mul_mat_close, cores, oracle_mul_mat

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import quantized_block_q4_gb300 as gq
else:  # collected on CPU machines, never run there (marked gpu)
    gq = None


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


def _static():
    return {gq.GQ_OPT_X_STATIC: 1, gq.GQ_OPT_WEIGHTS_STATIC: 1}


# (M, K, N, wide tokens): one token; several tokens of a batch (others
# normal); two n8 token tiles; K spanning several x chunks (N = 12, K = 8192).
CASES = [(1000, 4096, 1, [0]), (700, 11008, 1, [0]), (530, 4096, 5, [1, 3]), (300, 4096, 12, [0, 11]),
         (260, 8192, 12, [5]), (129, 1024, 8, list(range(8)))]


@pytest.mark.parametrize("static", [0, 1])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:3])))
def test_q4_0_decode_wide_range_x(case, static):
    M, K, N, wide = case
    W = synth.q4_0_weights(M, K, seed=15000 + M + N)
    X = synth.wide_range_activations(N, K, 15001 + M + N, wide)

    def run():
        y = gq.mul_mat_q4_0(dev(W), dev(X))
        torch.cuda.synchronize()
        gq.gq_sync_status()
        return y.cpu().numpy()
    y = _with_options(_static() if static else {}, run)
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    assert np.isfinite(y).all()
    assert_mul_mat_close(y, y_ref, s_ref, f"wide x M={M} K={K} N={N} static={static}")


def test_q4_0_decode_extreme_magnitudes():
    """Blocks up to 1e30 (the partial sums stay finite in fp32) next to
    ordinary tokens, and a token of tiny values (1e-30, no scaling)."""
    M, K, N = 400, 4096, 3
    W = synth.q4_0_weights(M, K, seed=15100)
    X = synth.wide_range_activations(N, K, 15101, [0], magnitudes=(1e20, 1e30))
    X[2] *= np.float32(1e-30)
    y = gq.mul_mat_q4_0(dev(W), dev(X)).cpu().numpy()
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    assert np.isfinite(y).all()
    assert_mul_mat_close(y, y_ref, s_ref, "extreme magnitudes")


@pytest.mark.parametrize("qtype", [1, 2], ids=["q4_1", "q8_0"])
@pytest.mark.parametrize("N", [1, 4, 12])
def test_legacy_decode_wide_range_x(qtype, N):
    M, K = 600, 4096
    W = synth.typed_weights(qtype, M, K, seed=15200 + N + qtype)
    X = synth.wide_range_activations(N, K, 15201 + N + qtype, [0, N - 1])
    y = gq.mul_mat(qtype, dev(W), dev(X)).cpu().numpy()
    y_ref, s_ref = oracle.get().mul_mat_typed(qtype, W, M, K, X, nthreads=cores())
    assert_mul_mat_close(y, y_ref, s_ref, f"wide x type {qtype} N={N}")


def test_mul_mat_id_decode_wide_range_x():
    E, M, K, T, S = 8, 512, 2048, 4, 2
    W = synth.moe_weights(E, M, K, 15300)
    X = synth.wide_range_activations(T * S, K, 15301, [2, 5]).reshape(T, S, K)
    ids = synth.expert_ids(T, S, E, 15302)
    old = gq.gq_get_option(gq.GQ_OPT_MOE_PATH)
    gq.gq_set_option(gq.GQ_OPT_MOE_PATH, 1)  # decode groups
    try:
        y = gq.mul_mat_id_q4_0(dev(W), E, dev(X), dev(ids))
        torch.cuda.synchronize()
        gq.gq_sync_status()
    finally:
        gq.gq_set_option(gq.GQ_OPT_MOE_PATH, old)
    y_ref, s_ref = oracle.get().mul_mat_id(W, E, M, K, X, ids, nthreads=cores())
    assert_mul_mat_close(y.cpu().numpy(), y_ref, s_ref, "MUL_MAT_ID decode, wide x")


@pytest.mark.parametrize("N", [1, 6])
def test_prepared_decode_wide_range_x(N):
    M, K = 300, 2880
    W = synth.q4_0_weights(M, K, seed=15400 + N)
    X = synth.wide_range_activations(N, K, 15401 + N, [0])
    Wp = gq.prepare_q4_0(dev(W), K)
    y = gq.mul_mat_q4_0_prepared(Wp, dev(X)).cpu().numpy()
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    assert_mul_mat_close(y, y_ref, s_ref, f"prepared, wide x N={N}")


def test_ordinary_x_unchanged_by_the_scaling_path():
    """A batch where only one token is wide: the other tokens' outputs are
    bit-identical to the same tokens computed without the wide one."""
    M, K, N = 500, 4096, 4
    W = dev(synth.q4_0_weights(M, K, seed=15500))
    X = synth.wide_range_activations(N, K, 15501, [2])
    Xn = X.copy()
    Xn[2] = 0.0
    a = gq.mul_mat_q4_0(W, dev(X)).cpu().numpy()
    b = gq.mul_mat_q4_0(W, dev(Xn)).cpu().numpy()
    keep = [0, 1, 3]
    assert np.array_equal(a[keep], b[keep])
