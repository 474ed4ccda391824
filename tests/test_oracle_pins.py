"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import numpy as np
import pytest

import oracle
import synth
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_threads_do_not_change_results(orc):
    M, K, N = 37, 288, 3
    W = synth.q4_0_weights(M, K, seed=5)
    X = synth.activations(N, K, seed=6)
    Y1, S1 = orc.mul_mat(W, M, K, X, nthreads=1)
    Y4, S4 = orc.mul_mat(W, M, K, X, nthreads=4)
    assert np.array_equal(Y1, Y4) and np.array_equal(S1, S4)


def test_empty_shapes(orc):
    W = np.zeros(0, dtype=np.uint8)
    Y, S = orc.mul_mat(W, 0, 64, np.zeros((2, 64), np.float32))
    assert Y.shape == (2, 0)
    W = synth.q4_0_weights(3, 32, seed=1)
    Y, S = orc.mul_mat(W, 3, 32, np.zeros((0, 32), np.float32))
    assert Y.shape == (0, 3)


def test_tolerance_helper():
    y_ref = np.array([1.0, -2.0, 0.0])
    s_ref = np.array([10.0, 10.0, 0.0])
    ok, worst = oracle.within_tolerance(y_ref + [0.0099, -0.0099, 9e-6], y_ref, s_ref)
    assert ok and worst < 1.0
    ok, _ = oracle.within_tolerance(y_ref + [0.0102, 0, 0], y_ref, s_ref)
    assert not ok
    ok, _ = oracle.within_tolerance([np.nan, -2.0, 0.0], y_ref, s_ref)
    assert not ok


def test_synth_is_deterministic():
    a = synth.q4_0_weights(4, 64, seed=9)
    b = synth.q4_0_weights(4, 64, seed=9)
    c = synth.q4_0_weights(4, 64, seed=10)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    d = a.reshape(4, 2, 18)[:, :, 0:2].copy().view("<f2").astype(np.float64)
    assert (d >= 0.005 - 1e-5).all() and (d <= 0.02 + 1e-5).all()
    x = synth.activations(3, 64, seed=9)
    assert x.dtype == np.float32 and x.shape == (3, 64)
