"""The timeout path of the bounded waits, made to run out on purpose.

Every in-kernel wait on an mbarrier gives up after GQ_OPT_WAIT_LIMIT_NS; the
kernel then sets the device error word, drains the copies and MMAs it issued,
releases tensor memory and returns, and gq_sync_status() reports
GQ_ERR_DEVICE_TIMEOUT (the library's counterpart of a failed ggml_status).
GQ_OPT_TEST_DROP_ARRIVE leaves one W copy of CTA 0 unissued, so that the
stage's consumers wait out the limit (1 ms here): a wait that nothing
completes, not a fault.  A normal call right after must match the oracle,
which shows the device and the library are usable again.
"""
import numpy as np
import pytest

import synth
from gpu_util import assert_mul_mat_close, oracle_mul_mat

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import quantized_block_q4_gb300 as gq
else:  # collected on CPU machines, never run there (marked gpu)
    gq = None


def _timeout_then_normal(drop, M, K, N, seed):
    W = synth.q4_0_weights(M, K, seed=seed)
    X = synth.activations(N, K, seed=seed + 1)
    Wd, Xd = torch.from_numpy(W).cuda(), torch.from_numpy(X).cuda()
    gq.gq_sync_status()  # nothing pending from earlier tests
    old = {k: gq.gq_get_option(k) for k in (gq.GQ_OPT_WAIT_LIMIT_NS, gq.GQ_OPT_TEST_DROP_ARRIVE)}
    try:
        gq.gq_set_option(gq.GQ_OPT_WAIT_LIMIT_NS, 1_000_000)
        gq.gq_set_option(gq.GQ_OPT_TEST_DROP_ARRIVE, drop)
        Y = torch.empty(N, M, device="cuda")
        gq.gq_mul_mat_q4_0(Wd, M, K, Xd, N, Y)
        with pytest.raises(gq.GQError) as e:
            gq.gq_sync_status()
        assert e.value.status == gq.GQ_ERR_DEVICE_TIMEOUT, str(e.value)
    finally:
        for k, v in old.items():
            gq.gq_set_option(k, v)
    gq.gq_sync_status()  # the error word was read and cleared
    Y = gq.mul_mat_q4_0(Wd, Xd)
    gq.gq_sync_status()
    y_ref, s_ref = oracle_mul_mat(W, M, K, X)
    assert_mul_mat_close(Y.cpu().numpy(), y_ref, s_ref, f"normal call after the timeout (drop={drop})")


def test_decode_kernel_timeout_path():
    _timeout_then_normal(1, 1000, 4096, 1, 18000)


def test_decode_kernel_timeout_path_batch():
    _timeout_then_normal(1, 600, 4096, 6, 18010)


def test_tensor_core_kernel_timeout_path():
    _timeout_then_normal(2, 700, 4096, 64, 18020)
