"""The allocation-free MUL_MAT entry point (gq_mul_mat_q4_0_noalloc).

Callers that cannot let a library allocate device memory (a memory pool that
owns the whole device, a fixed arena, an allocation-free hot loop) use this
entry point; it keeps the bf16 copy of the activations in a fixed array inside
the library.  This test calls it through the C ABI twice in a row, on
different shapes, and checks each result against the allocating entry point
gq_mul_mat_q4_0 and the oracle, with the tolerance every MUL_MAT test uses.
It sits in its own file, collected last, and passes alone in a fresh process
as well as after the other tests.
"""
import numpy as np
import pytest

import synth
from gpu_util import assert_mul_mat_close, oracle_mul_mat

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _run_both(gq, M, K, N, seed):
    W = synth.q4_0_weights(M, K, seed=seed)
    X = synth.activations(N, K, seed=seed + 1)
    Wd, Xd = torch.from_numpy(W).cuda(), torch.from_numpy(X).cuda()
    y_new = torch.full((N, M), float("nan"), device="cuda")
    y_old = torch.full((N, M), float("nan"), device="cuda")
    gq.gq_mul_mat_q4_0_noalloc(Wd, M, K, Xd, N, y_new)
    gq.gq_mul_mat_q4_0(Wd, M, K, Xd, N, y_old)
    torch.cuda.synchronize()
    gq.gq_sync_status()
    return W, X, y_new.cpu().numpy(), y_old.cpu().numpy()


@pytest.mark.parametrize("N", [1, 7, 16, 70, 512])
def test_noalloc_token_counts(N):
    """One partial token tile (N = 1, 7, 16) up to two full 256-token tiles."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import quantized_block_q4_gb300 as gq
    M, K = 640, 2048
    W, X, y_new, y_old = _run_both(gq, M, K, N, 90 + N)
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    assert_mul_mat_close(y_new, y_ref, s_ref, f"noalloc vs oracle N={N}")
    assert_mul_mat_close(y_new, y_old, s_ref, f"noalloc vs gq_mul_mat_q4_0 N={N}")


def test_noalloc_x_and_y_four_byte_aligned():
    """X and Y one float past a 16-byte boundary (the entry point accepts
    4-byte alignment for both)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import quantized_block_q4_gb300 as gq
    M, K, N = 333, 1024, 9
    W = synth.q4_0_weights(M, K, seed=95)
    X = synth.activations(N, K, seed=96)
    Wd = torch.from_numpy(W).cuda()
    xbuf = torch.zeros(N * K + 4, device="cuda")
    xbuf[1:1 + N * K] = torch.from_numpy(X).cuda().reshape(-1)
    ybuf = torch.full((N * M + 4,), float("nan"), device="cuda")
    gq.gq_mul_mat_q4_0_noalloc(Wd, M, K, xbuf.data_ptr() + 4, N, ybuf.data_ptr() + 4)
    torch.cuda.synchronize()
    gq.gq_sync_status()
    out = ybuf.cpu().numpy()
    y = out[1:1 + N * M].reshape(N, M)
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    assert_mul_mat_close(y, y_ref, s_ref, "noalloc with X and Y offset by one float")
    assert np.isnan(out[0]) and np.isnan(out[1 + N * M:]).all()  # nothing written outside Y


def test_noalloc_matches_allocating_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import quantized_block_q4_gb300 as gq
    # first call: larger N*K; second call: smaller, so stale contents of the
    # shared array from the first call would show up if they were ever read
    for (M, K, N, seed) in [(1000, 4096, 512, 81), (300, 1024, 70, 82)]:
        W, X, y_new, y_old = _run_both(gq, M, K, N, seed)
        y_ref, s_ref = oracle_mul_mat(W, M, K, X)
        assert_mul_mat_close(y_new, y_old, s_ref, f"noalloc vs gq_mul_mat_q4_0 M={M} K={K} N={N}")
        assert_mul_mat_close(y_new, y_ref, s_ref, f"noalloc vs oracle M={M} K={K} N={N}")


def test_noalloc_rejects_oversize_and_bad_shapes():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import quantized_block_q4_gb300 as gq
    W = torch.zeros(18 * 8, dtype=torch.uint8, device="cuda")
    X = torch.zeros(1, dtype=torch.float32, device="cuda")
    Y = torch.zeros(1, dtype=torch.float32, device="cuda")
    with pytest.raises(gq.GQError) as e:      # N*K beyond the fixed array; rejected before any access
        gq.gq_mul_mat_q4_0_noalloc(W, 1, 8192, X, 1024, Y)
    assert e.value.status == gq.GQ_ERR_SHAPE and "exceeds" in str(e.value)
    with pytest.raises(gq.GQError) as e:
        gq.gq_mul_mat_q4_0_noalloc(W, 1, 288, X, 1, Y)
    assert e.value.status == gq.GQ_ERR_SHAPE


def test_noalloc_rejects_alignment_and_null_and_accepts_empty():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import quantized_block_q4_gb300 as gq
    W = torch.zeros(18 * 8 * 2 + 16, dtype=torch.uint8, device="cuda")
    X = torch.ones(256, dtype=torch.float32, device="cuda")
    Y = torch.full((4,), 7.0, device="cuda")
    with pytest.raises(gq.GQError) as e:      # W two bytes past a 16-byte boundary
        gq.gq_mul_mat_q4_0_noalloc(W.data_ptr() + 2, 1, 256, X, 1, Y)
    assert e.value.status == gq.GQ_ERR_ALIGN
    with pytest.raises(gq.GQError) as e:
        gq.gq_mul_mat_q4_0_noalloc(W, 1, 256, 0, 1, Y)
    assert e.value.status == gq.GQ_ERR_NULL
    gq.gq_mul_mat_q4_0_noalloc(W, 1, 256, X, 0, Y)  # N = 0: nothing to do
    gq.gq_mul_mat_q4_0_noalloc(W, 0, 256, X, 1, Y)  # M = 0: nothing to do
    torch.cuda.synchronize()
    assert (Y.cpu().numpy() == 7.0).all()
    assert gq.gq_last_error() == ""  # a successful call leaves no stale message
