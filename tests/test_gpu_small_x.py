"""Activations far below 1 on the decode kernel, against the oracle.

The decode kernel stages x as fp16 (x for the low nibbles, x/16 for the high
ones).  Values below 2^-14 would fall on fp16's subnormal grid and lose
significant bits, so a warp's chunk of a token whose largest |x| is below
2^-10 is staged times an exact power of two and its partial sums scaled back.
With O(1) weights (d ~ U[0.5, 2]) the relative error term dominates the
1e-5 absolute term of |y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-5, so these
cases check the precision of the small-x path itself.  Inputs: N(0, 1)
activations times 1e-5 or 1e-7 (fp32, exact scaling of the seeded draws).
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

D_RANGE = (0.5, 2.0)  # fp16 block scales of O(1) weights


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


def small_x(N, K, seed, scale):
    return synth.activations(N, K, seed) * np.float32(scale)


def _check_q4_0(M, K, N, scale, seed, label, opts=None):
    W = synth.q4_0_weights(M, K, seed=seed, d_range=D_RANGE)
    X = small_x(N, K, seed + 1, scale)

    def run():
        y = gq.mul_mat_q4_0(dev(W), dev(X))
        torch.cuda.synchronize()
        gq.gq_sync_status()
        return y.cpu().numpy()
    y = _with_options(opts or {}, run)
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    assert np.isfinite(y).all()
    return assert_mul_mat_close(y, y_ref, s_ref, label)


@pytest.mark.parametrize("scale", [1e-5, 1e-7])
@pytest.mark.parametrize("N", [1, 4, 12])
@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
def test_q4_0_decode_small_x(variant, N, scale):
    M, K = 700, 4096
    _check_q4_0(M, K, N, scale, 16000 + 10 * variant + N, f"small x {scale} N={N} variant={variant}",
                {gq.GQ_OPT_DECODE_VARIANT: variant})


@pytest.mark.parametrize("N", [1, 3])
@pytest.mark.parametrize("static", [0, 1])
@pytest.mark.parametrize("shape", [(11008, 4096), (4096, 11008)])
def test_q4_0_decode_small_x_sweep_shapes(shape, static, N):
    """The sweep's shapes at 1 and 3 tokens, with and without the static
    promises (the 4-warp and 8-warp CTA layouts)."""
    M, K = shape
    opts = {gq.GQ_OPT_X_STATIC: static, gq.GQ_OPT_WEIGHTS_STATIC: static}
    _check_q4_0(M, K, N, 1e-6, 16100 + M + static + N, f"small x {M}x{K} N={N} static={static}", opts)


@pytest.mark.parametrize("qtype", [1, 2], ids=["q4_1", "q8_0"])
@pytest.mark.parametrize("N", [1, 4, 12])
def test_legacy_decode_small_x(qtype, N):
    M, K = 600, 4096
    W = synth.typed_weights(qtype, M, K, seed=16200 + N + qtype, d_scale=100.0)
    X = small_x(N, K, 16201 + N + qtype, 1e-6)
    y = gq.mul_mat(qtype, dev(W), dev(X)).cpu().numpy()
    y_ref, s_ref = oracle.get().mul_mat_typed(qtype, W, M, K, X, nthreads=cores())
    assert_mul_mat_close(y, y_ref, s_ref, f"small x type {qtype} N={N}")


@pytest.mark.parametrize("T", [1, 4])
def test_mul_mat_id_decode_small_x(T):
    E, M, K, S = 8, 512, 2048, 2
    W = np.concatenate([synth.q4_0_weights(M, K, 16300 + 7919 * e, D_RANGE) for e in range(E)], axis=0)
    X = small_x(T * S, K, 16301 + T, 1e-6).reshape(T, S, K)
    ids = synth.expert_ids(T, S, E, 16302 + T)
    old = gq.gq_get_option(gq.GQ_OPT_MOE_PATH)
    gq.gq_set_option(gq.GQ_OPT_MOE_PATH, 1)  # decode groups
    try:
        y = gq.mul_mat_id_q4_0(dev(W), E, dev(X), dev(ids))
        torch.cuda.synchronize()
        gq.gq_sync_status()
    finally:
        gq.gq_set_option(gq.GQ_OPT_MOE_PATH, old)
    y_ref, s_ref = oracle.get().mul_mat_id(W, E, M, K, X, ids, nthreads=cores())
    assert_mul_mat_close(y.cpu().numpy(), y_ref, s_ref, f"MUL_MAT_ID decode, small x, T={T}")


@pytest.mark.parametrize("N", [1, 6])
def test_prepared_decode_small_x(N):
    M, K = 300, 2880
    W = synth.q4_0_weights(M, K, seed=16400 + N, d_range=D_RANGE)
    X = small_x(N, K, 16401 + N, 1e-6)
    Wp = gq.prepare_q4_0(dev(W), K)
    y = gq.mul_mat_q4_0_prepared(Wp, dev(X)).cpu().numpy()
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    assert_mul_mat_close(y, y_ref, s_ref, f"prepared, small x N={N}")


def test_tiny_token_beside_ordinary_ones():
    """One tiny token in a batch of ordinary ones: every token is within
    tolerance, and the ordinary tokens' outputs are bit-identical to the same
    batch with the tiny token set to zero (its scaling touches no other token)."""
    M, K, N = 500, 4096, 4
    W = synth.q4_0_weights(M, K, seed=16500, d_range=D_RANGE)
    X = synth.activations(N, K, 16501)
    X[2] *= np.float32(1e-7)
    Xn = X.copy()
    Xn[2] = 0.0
    Wd = dev(W)
    a = gq.mul_mat_q4_0(Wd, dev(X)).cpu().numpy()
    b = gq.mul_mat_q4_0(Wd, dev(Xn)).cpu().numpy()
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    assert_mul_mat_close(a, y_ref, s_ref, "tiny token in an ordinary batch")
    keep = [0, 1, 3]
    assert np.array_equal(a[keep], b[keep])
