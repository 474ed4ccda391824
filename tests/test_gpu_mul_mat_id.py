"""MUL_MAT_ID (expert-routed Q4_0 matmul) on the GPU against the oracle.

Every element must satisfy |y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-5, with
y_ref and the sum from the fp64 oracle; rows of out-of-range ids must be NaN
on both sides.  Each path is checked on its own (decode kernel, tensor-core
kernel, generic kernel) and through the default dispatch.  Inputs: synth.py.
"""
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

AUTO, DECODE, TC, GENERIC = "auto", "decode", "tc", "generic"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class _path:
    def __init__(self, path):
        self.path = path

    def __enter__(self):
        self.old = (gq.gq_get_option(gq.GQ_OPT_MOE_PATH), gq.gq_get_option(gq.GQ_OPT_FORCE_GENERIC))
        gq.gq_set_option(gq.GQ_OPT_MOE_PATH, {AUTO: 0, DECODE: 1, TC: 2, GENERIC: 0}[self.path])
        gq.gq_set_option(gq.GQ_OPT_FORCE_GENERIC, 1 if self.path == GENERIC else 0)

    def __exit__(self, *a):
        gq.gq_set_option(gq.GQ_OPT_MOE_PATH, self.old[0])
        gq.gq_set_option(gq.GQ_OPT_FORCE_GENERIC, self.old[1])


def gpu_mul_mat_id(W, E, X, ids, path=AUTO):
    with _path(path):
        Y = gq.mul_mat_id_q4_0(dev(W), E, dev(X), dev(ids))
        torch.cuda.synchronize()
    return Y.cpu().numpy()


def check(E, M, K, T, S, seed, path=AUTO, skew=0.0, ids=None, label=""):
    W = synth.moe_weights(E, M, K, seed)
    X = synth.activations(T * S, K, seed + 1).reshape(T, S, K)
    if ids is None:
        ids = synth.expert_ids(T, S, E, seed + 2, skew)
    y = gpu_mul_mat_id(W, E, X, ids, path)
    gq.gq_sync_status()
    y_ref, s_ref = oracle.get().mul_mat_id(W, E, M, K, X, ids, nthreads=cores())
    return assert_mul_mat_close(y, y_ref, s_ref, label or f"E={E} M={M} K={K} T={T} S={S} {path}")


# (E, M, K, T, S): decode-sized batches, prefill-sized batches, ragged M (not a
# multiple of the 16/32/128-row tiles), K spanning several 256-k chunks.
SHAPES = [
    (8, 512, 1024, 1, 2),
    (8, 1000, 512, 3, 2),
    (8, 384, 768, 16, 2),
    (64, 256, 512, 4, 8),
    (8, 300, 1024, 64, 2),
    (8, 1000, 1024, 512, 2),
    (4, 130, 512, 300, 4),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("path", [AUTO, DECODE, TC])
def test_mul_mat_id_matches_oracle(shape, path):
    E, M, K, T, S = shape
    check(E, M, K, T, S, seed=12000 + sum(shape), path=path)


@pytest.mark.parametrize("path", [DECODE, TC])
def test_skewed_routing(path):
    """Zipf-like routing: the first experts take most tokens (several decode
    groups and several 256-token tiles for one expert), most take few or none."""
    check(32, 400, 512, 700, 4, seed=12100, path=path, skew=1.5)


@pytest.mark.parametrize("path", [DECODE, TC])
def test_every_pair_to_one_expert(path):
    E, M, K, T, S = 8, 260, 512, 200, 2
    ids = np.full((T, S), 5, dtype=np.int32)
    check(E, M, K, T, S, seed=12200, path=path, ids=ids)


@pytest.mark.parametrize("path", [AUTO, DECODE, TC])
def test_single_pair_and_single_expert(path):
    check(1, 200, 256, 1, 1, seed=12300, path=path)
    check(1, 129, 512, 40, 1, seed=12301, path=path)


@pytest.mark.parametrize("path", [DECODE, TC])
def test_many_experts_few_tokens(path):
    """More experts than pairs: most experts unused, each used one by one pair."""
    check(300, 64, 256, 5, 6, seed=12400, path=path)


def test_more_decode_groups_than_ctas():
    """About 280 used experts with a few tokens each: more decode groups than
    the launch has CTAs, so CTAs run several groups one after the other."""
    check(300, 64, 256, 100, 6, seed=12401, path=DECODE)


def test_generic_path_odd_shapes():
    """K % 256 != 0 (generic kernel by shape) and the forced generic kernel."""
    check(8, 77, 96, 5, 2, seed=12500)
    check(8, 300, 512, 9, 2, seed=12501, path=GENERIC)


@pytest.mark.parametrize("path", [DECODE, TC, GENERIC])
def test_out_of_range_ids_give_nan_rows_and_status(path):
    E, M, K, T, S = 8, 256, 512, 20, 2
    W = synth.moe_weights(E, M, K, 12600)
    X = synth.activations(T * S, K, 12601).reshape(T, S, K)
    ids = synth.expert_ids(T, S, E, 12602)
    ids[3, 1] = E
    ids[7, 0] = -1
    ids[19, 1] = 1 << 30
    with _path(path):
        y = gq.mul_mat_id_q4_0(dev(W), E, dev(X), dev(ids))
        with pytest.raises(gq.GQError) as e:
            gq.gq_sync_status()
    assert e.value.status == gq.GQ_ERR_BAD_INDEX
    gq.gq_sync_status()  # cleared
    y = y.cpu().numpy()
    y_ref, s_ref = oracle.get().mul_mat_id(W, E, M, K, X, ids, nthreads=cores())
    bad = np.isnan(y_ref).all(axis=-1)
    assert bad.sum() == 3
    assert np.isnan(y[bad]).all(), "rows of bad ids must be NaN"
    assert_mul_mat_close(y[~bad], y_ref[~bad], s_ref[~bad], f"good rows, {path}")


@pytest.mark.parametrize("path", [DECODE, TC])
def test_repeatable_bit_for_bit(path):
    E, M, K, T, S = 8, 512, 1024, 96, 2
    W = dev(synth.moe_weights(E, M, K, 12700))
    X = dev(synth.activations(T * S, K, 12701).reshape(T, S, K))
    ids = dev(synth.expert_ids(T, S, E, 12702))
    with _path(path):
        a = gq.mul_mat_id_q4_0(W, E, X, ids)
        b = gq.mul_mat_id_q4_0(W, E, X, ids)
        torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_k_zero_and_empty():
    E, M, T, S = 4, 64, 3, 2
    ids = dev(np.array([[0, 1], [2, 9], [3, 3]], dtype=np.int32))
    Y = torch.full((T, S, M), 7.0, device="cuda")
    gq.gq_mul_mat_id_q4_0(None, E, M, 0, None, S, ids, T, Y)
    with pytest.raises(gq.GQError):
        gq.gq_sync_status()
    y = Y.cpu().numpy()
    assert np.isnan(y[1, 1]).all()
    y[1, 1] = 0
    assert not y.any(), "K = 0 must write zeros"
    gq.gq_mul_mat_id_q4_0(None, E, M, 256, None, S, ids, 0, None)  # T = 0: no-op


def test_full_size_sampled_pairs():
    """The prefill-sized workload (8 experts of 14336 x 4096, 512 tokens x 2
    slots): the GPU computes every pair; the oracle checks a sample of pairs,
    which by definition do not depend on one another."""
    E, M, K, T, S = 8, 14336, 4096, 512, 2
    W = synth.moe_weights(E, M, K, 12800)
    X = synth.activations(T * S, K, 12801).reshape(T, S, K)
    ids = synth.expert_ids(T, S, E, 12802)
    y = gpu_mul_mat_id(W, E, X, ids)
    gq.gq_sync_status()
    pick = np.random.default_rng(12803).choice(T, 6, replace=False)
    y_ref, s_ref = oracle.get().mul_mat_id(W, E, M, K, X[pick], ids[pick], nthreads=cores())
    assert_mul_mat_close(y[pick], y_ref, s_ref, "full size, sampled tokens")


def test_decode_full_size():
    """Decode-sized batch on full-size experts: 4 tokens x 2 slots."""
    E, M, K, T, S = 8, 14336, 4096, 4, 2
    check(E, M, K, T, S, seed=12900)


@pytest.mark.parametrize("path", [DECODE, TC])
def test_single_token_repeated_expert(path):
    """One token whose slots name the same expert twice (and a third slot
    another): the single-token decode path runs one group per slot."""
    ids = np.array([[3, 3, 5]], dtype=np.int32)
    check(8, 700, 1024, 1, 3, seed=12950, path=path, ids=ids)


def test_single_token_many_slots():
    check(64, 512, 2048, 1, 8, seed=12960, path=DECODE)


def test_single_token_bad_ids_direct_groups():
    """A single token reads its ids in the decode kernel itself (no routing
    kernel): out-of-range slots give NaN rows and GQ_ERR_BAD_INDEX, the
    others match the oracle."""
    E, M, K, T, S = 8, 700, 1024, 1, 5
    W = synth.moe_weights(E, M, K, 12970)
    X = synth.activations(T * S, K, 12971).reshape(T, S, K)
    ids = np.array([[3, E, -1, 5, 3]], dtype=np.int32)
    with _path(DECODE):
        y = gq.mul_mat_id_q4_0(dev(W), E, dev(X), dev(ids))
        with pytest.raises(gq.GQError) as e:
            gq.gq_sync_status()
    assert e.value.status == gq.GQ_ERR_BAD_INDEX
    gq.gq_sync_status()  # cleared
    y = y.cpu().numpy()
    y_ref, s_ref = oracle.get().mul_mat_id(W, E, M, K, X, ids, nthreads=cores())
    bad = np.isnan(y_ref).all(axis=-1)
    assert bad.sum() == 2 and bad[0, 1] and bad[0, 2]
    assert np.isnan(y[bad]).all(), "rows of bad ids must be NaN"
    assert_mul_mat_close(y[~bad], y_ref[~bad], s_ref[~bad], "single token, good slots")


@pytest.mark.parametrize("path", [AUTO, DECODE])
def test_single_token_full_size_experts(path):
    """1 token x 2 slots on full-size experts (the single-token decode case)."""
    check(8, 14336, 4096, 1, 2, seed=12980, path=path)
