"""Pins of the oracle's MUL_MAT_ID (expert-routed MUL_MAT; the MUL_MAT_ID probe
of "GGUF loading, mmap and tensor placement", step six) against facts other
than itself: the one-expert case is MUL_MAT, relabelling the experts does not
change Y, a one-hot x selects a dequantised column of the chosen expert, and a
dense fp64 computation on tiny inputs agrees."""
import os
import shutil

import numpy as np
import pytest

import oracle
import synth


def _inputs(E, M, K, T, S, seed):
    W = np.concatenate([synth.q4_0_weights(M, K, seed=seed + e) for e in range(E)], axis=0)
    X = synth.activations(T * S, K, seed=seed + 100).reshape(T, S, K)
    ids = np.random.Generator(np.random.SFC64(seed + 200)).integers(0, E, (T, S)).astype(np.int32)
    return W, X, ids


def pin_one_expert_is_mul_mat(orc):
    M, K, T, S = 37, 256, 3, 4
    W, X, _ = _inputs(1, M, K, T, S, 9000)
    ids = np.zeros((T, S), dtype=np.int32)
    Y, Sa = orc.mul_mat_id(W, 1, M, K, X, ids)
    Y2, S2 = orc.mul_mat(W, M, K, X.reshape(T * S, K))
    assert np.array_equal(Y.reshape(T * S, M), Y2) and np.array_equal(Sa.reshape(T * S, M), S2)


def pin_relabelled_experts_give_the_same_result(orc):
    E, M, K, T, S = 5, 24, 128, 4, 3
    W, X, ids = _inputs(E, M, K, T, S, 9100)
    perm = np.array([3, 0, 4, 1, 2])
    blocks = W.reshape(E, M, -1)
    Wp = np.empty_like(blocks)
    Wp[perm] = blocks                      # expert e moves to slot perm[e]
    Y1, _ = orc.mul_mat_id(W, E, M, K, X, ids)
    Y2, _ = orc.mul_mat_id(Wp.reshape(E * M, -1), E, M, K, X, perm[ids].astype(np.int32))
    assert np.array_equal(Y1, Y2)


def pin_one_hot_selects_expert_column(orc):
    E, M, K, T, S = 4, 16, 128, 2, 4
    W, _, ids = _inputs(E, M, K, T, S, 9200)
    ks = np.random.Generator(np.random.SFC64(9201)).integers(0, K, (T, S))
    X = np.zeros((T, S, K), dtype=np.float32)
    for t in range(T):
        for s in range(S):
            X[t, s, ks[t, s]] = 1.0
    Y, _ = orc.mul_mat_id(W, E, M, K, X, ids)
    dense = orc.dequant(W, E * M, K).reshape(E, M, K)
    for t in range(T):
        for s in range(S):
            assert np.array_equal(Y[t, s], dense[ids[t, s], :, ks[t, s]].astype(np.float64))


def pin_dense_brute_force(orc):
    E, M, K, T, S = 3, 5, 64, 3, 2
    W, X, ids = _inputs(E, M, K, T, S, 9300)
    dense = orc.dequant(W, E * M, K).reshape(E, M, K).astype(np.float64)
    Y, Sa = orc.mul_mat_id(W, E, M, K, X, ids)
    ref = np.einsum("tsmk,tsk->tsm", dense[ids], X.astype(np.float64))
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(Sa, np.einsum("tsmk,tsk->tsm", np.abs(dense[ids]), np.abs(X.astype(np.float64))),
                       rtol=1e-12, atol=1e-12)


def pin_out_of_range_id_gives_nan_rows(orc):
    E, M, K, T, S = 2, 8, 64, 1, 3
    W, X, ids = _inputs(E, M, K, T, S, 9400)
    ids[0, 1] = 7
    Y, _ = orc.mul_mat_id(W, E, M, K, X, ids)
    assert np.isnan(Y[0, 1]).all() and not np.isnan(Y[0, 0]).any() and not np.isnan(Y[0, 2]).any()


ID_PINS = [pin_one_expert_is_mul_mat, pin_relabelled_experts_give_the_same_result, pin_one_hot_selects_expert_column,
           pin_dense_brute_force, pin_out_of_range_id_gives_nan_rows]


@pytest.mark.parametrize("pin", ID_PINS, ids=lambda p: p.__name__)
def test_mul_mat_id_pin(pin, orc):
    pin(orc)


ID_MUTATIONS = {
    "ids_transposed": [("int32_t e = ids[t * S + s];", "int32_t e = ids[s * T + t];")],
    "wrong_expert": [("oracle_mul_mat_q4_0(W + (size_t)e * expert_bytes,",
                      "oracle_mul_mat_q4_0(W + (size_t)(e ? e - 1 : 0) * expert_bytes,")],
    "x_of_other_slot": [("X + (size_t)(t * S + s) * (size_t)K, 1,", "X + (size_t)(s * T + t) * (size_t)K, 1,")],
    "bad_id_not_flagged": [("if (e < 0 || e >= n_expert) {", "if (e < 0) {")],
}


@pytest.mark.parametrize("name", sorted(ID_MUTATIONS))
def test_mul_mat_id_mutation_is_caught(name, tmp_path):
    src = open(oracle.SRC).read()
    for old, new in ID_MUTATIONS[name]:
        assert old in src, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new)
    if name == "bad_id_not_flagged":    # keep the mutant in bounds: clamp instead of reading past W
        src = src.replace("oracle_mul_mat_q4_0(W + (size_t)e * expert_bytes,",
                          "oracle_mul_mat_q4_0(W + (size_t)(e < n_expert ? e : n_expert - 1) * expert_bytes,")
    mdir = tmp_path / "src"
    mdir.mkdir()
    (mdir / "q4_0_oracle.c").write_text(src)
    shutil.copy(oracle.HDR, mdir / "q4_0_oracle.h")
    lib = oracle.build_library(str(mdir / "q4_0_oracle.c"), str(tmp_path / "libmut.so"), include_dir=str(mdir))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in ID_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutation {name}"
    os.remove(lib)
