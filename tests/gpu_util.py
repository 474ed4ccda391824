"""Helpers shared by the GPU parity tests (marshalling and comparison only)."""
from __future__ import annotations

import os

import numpy as np

import oracle


def cores() -> int:
    return max(1, os.cpu_count() or 1)


def oracle_mul_mat(W: np.ndarray, M: int, K: int, X: np.ndarray):
    return oracle.get().mul_mat(W, M, K, X, nthreads=cores())


def assert_mul_mat_close(y_gpu: np.ndarray, y_ref: np.ndarray, s_ref: np.ndarray, label: str = "") -> float:
    """|y - y_ref| <= 1e-3 * sum|w x| + 1e-5 element by element; returns the worst ratio."""
    ok, worst = oracle.within_tolerance(y_gpu, y_ref, s_ref)
    if not ok:
        bound = 1e-3 * s_ref + 1e-5
        ratio = np.abs(y_gpu - y_ref) / bound
        idx = np.unravel_index(np.nanargmax(np.where(np.isnan(ratio), np.inf, ratio)), ratio.shape)
        raise AssertionError(f"{label}: tolerance exceeded, worst ratio {worst:.3g} at {idx}: "
                             f"gpu={y_gpu[idx]!r} ref={y_ref[idx]!r} s={s_ref[idx]!r}")
    return worst
