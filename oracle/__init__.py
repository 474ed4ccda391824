"""CPU oracle for Q4_0 dequantisation and MUL_MAT -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs it.

The arithmetic lives in plain C (``q4_0_oracle.c``), compiled here with gcc
into ``oracle/_build/liboracle.so`` and called through ctypes.  See the C
header for what each function computes and which passage defines it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "q4_0_oracle.c")
HDR = os.path.join(_HERE, "q4_0_oracle.h")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
          "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None


def build_library(src: str = SRC, out: str = LIB_PATH, include_dir: str = _HERE) -> str:
    """Compile the oracle C source into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-I", include_dir, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR))


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, sz, vp, i32 = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
        lib.oracle_q4_0_nbytes.argtypes = [i64, i64]
        lib.oracle_q4_0_nbytes.restype = sz
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_half_to_float_n.argtypes = [vp, sz, vp]
        lib.oracle_half_to_float_n.restype = None
        lib.oracle_dequant_q4_0.argtypes = [vp, i64, i64, vp]
        lib.oracle_dequant_q4_0.restype = None
        lib.oracle_mul_mat_q4_0.argtypes = [vp, i64, i64, vp, i64, vp, vp, i32]
        lib.oracle_mul_mat_q4_0.restype = None
        lib.oracle_float_to_half.argtypes = [ctypes.c_float]
        lib.oracle_float_to_half.restype = ctypes.c_uint16
        lib.oracle_quantize_q4_0.argtypes = [vp, i64, i64, vp]
        lib.oracle_quantize_q4_0.restype = None
        lib.oracle_mul_mat_id_q4_0.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, vp, i32]
        lib.oracle_mul_mat_id_q4_0.restype = None
        lib.oracle_type_nbytes.argtypes = [i32, i64, i64]
        lib.oracle_type_nbytes.restype = sz
        lib.oracle_dequant_typed.argtypes = [i32, vp, i64, i64, vp]
        lib.oracle_dequant_typed.restype = None
        lib.oracle_mul_mat_typed.argtypes = [i32, vp, i64, i64, vp, i64, vp, vp, i32]
        lib.oracle_mul_mat_typed.restype = None
        lib.oracle_validate_typed.argtypes = [i32, vp, i64, i64, vp, vp]
        lib.oracle_validate_typed.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        self.lib = lib
        self.path = path

    # -- thin wrappers (argument marshalling only) --------------------------
    def nbytes(self, M: int, K: int) -> int:
        return int(self.lib.oracle_q4_0_nbytes(M, K))

    def half_to_double(self, h: int) -> float:
        return float(self.lib.oracle_half_to_double(h))

    def half_to_float(self, bits: np.ndarray) -> np.ndarray:
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(bits.shape, dtype=np.float32)
        self.lib.oracle_half_to_float_n(bits.ctypes.data, bits.size, out.ctypes.data)
        return out

    def dequant(self, W: np.ndarray, M: int, K: int) -> np.ndarray:
        W = np.ascontiguousarray(W, dtype=np.uint8)
        if W.size != self.nbytes(M, K):
            raise ValueError("W has the wrong number of bytes")
        out = np.empty((M, K), dtype=np.float32)
        self.lib.oracle_dequant_q4_0(W.ctypes.data, M, K, out.ctypes.data)
        return out

    def mul_mat(self, W: np.ndarray, M: int, K: int, X: np.ndarray,
                nthreads: int = 1):
        """Returns (Y, S), both fp64 [N][M]."""
        W = np.ascontiguousarray(W, dtype=np.uint8)
        X = np.ascontiguousarray(X, dtype=np.float32)
        if W.size != self.nbytes(M, K):
            raise ValueError("W has the wrong number of bytes")
        N = X.shape[0] if X.ndim == 2 else 1
        if X.size != N * K:
            raise ValueError("X must be [N][K]")
        Y = np.empty((N, M), dtype=np.float64)
        S = np.empty((N, M), dtype=np.float64)
        self.lib.oracle_mul_mat_q4_0(W.ctypes.data, M, K, X.ctypes.data, N,
                                     Y.ctypes.data, S.ctypes.data, int(nthreads))
        return Y, S

    def float_to_half(self, f: float) -> int:
        return int(self.lib.oracle_float_to_half(float(f)))

    def quantize(self, W: np.ndarray) -> np.ndarray:
        """fp32 W[M][K] -> uint8 [M][K/32*18] Q4_0 blocks."""
        W = np.ascontiguousarray(W, dtype=np.float32)
        M, K = W.shape
        if K % 32:
            raise ValueError("K must be a multiple of 32")
        out = np.empty((M, K // 32 * 18), dtype=np.uint8)
        self.lib.oracle_quantize_q4_0(W.ctypes.data, M, K, out.ctypes.data)
        return out

    def mul_mat_id(self, W: np.ndarray, n_expert: int, M: int, K: int, X: np.ndarray, ids: np.ndarray,
                   nthreads: int = 1):
        """W: n_expert*M rows of blocks; X [T][S][K] fp32; ids [T][S] int32 -> (Y, S) fp64 [T][S][M]."""
        W = np.ascontiguousarray(W, dtype=np.uint8)
        X = np.ascontiguousarray(X, dtype=np.float32)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        if W.size != n_expert * self.nbytes(M, K):
            raise ValueError("W has the wrong number of bytes")
        T, S = ids.shape
        if X.shape != (T, S, K):
            raise ValueError("X must be [T][S][K]")
        Y = np.empty((T, S, M), dtype=np.float64)
        Sa = np.empty((T, S, M), dtype=np.float64)
        self.lib.oracle_mul_mat_id_q4_0(W.ctypes.data, n_expert, M, K, X.ctypes.data, S, ids.ctypes.data, T,
                                        Y.ctypes.data, Sa.ctypes.data, int(nthreads))
        return Y, Sa

    def type_nbytes(self, qtype: int, M: int, K: int) -> int:
        return int(self.lib.oracle_type_nbytes(qtype, M, K))

    def dequant_typed(self, qtype: int, W: np.ndarray, M: int, K: int) -> np.ndarray:
        W = np.ascontiguousarray(W, dtype=np.uint8)
        if W.size != self.type_nbytes(qtype, M, K):
            raise ValueError("W has the wrong number of bytes")
        out = np.empty((M, K), dtype=np.float32)
        self.lib.oracle_dequant_typed(qtype, W.ctypes.data, M, K, out.ctypes.data)
        return out

    def mul_mat_typed(self, qtype: int, W: np.ndarray, M: int, K: int, X: np.ndarray, nthreads: int = 1):
        """Returns (Y, S), both fp64 [N][M]."""
        W = np.ascontiguousarray(W, dtype=np.uint8)
        X = np.ascontiguousarray(X, dtype=np.float32)
        if W.size != self.type_nbytes(qtype, M, K):
            raise ValueError("W has the wrong number of bytes")
        N = X.shape[0]
        Y = np.empty((N, M), dtype=np.float64)
        S = np.empty((N, M), dtype=np.float64)
        self.lib.oracle_mul_mat_typed(qtype, W.ctypes.data, M, K, X.ctypes.data, N, Y.ctypes.data,
                                      S.ctypes.data, int(nthreads))
        return Y, S

    def validate(self, qtype: int, W: np.ndarray, M: int, K: int):
        """(count, first): blocks with a non-finite scale, and the first one's
        flat index (row * K/32 + block; super-blocks of 256 for Q4_K), or None
        when there is none."""
        W = np.ascontiguousarray(W, dtype=np.uint8)
        if W.size != self.type_nbytes(qtype, M, K):
            raise ValueError("W has the wrong number of bytes")
        out = np.zeros(2, dtype=np.uint64)
        self.lib.oracle_validate_typed(qtype, W.ctypes.data, M, K, out.ctypes.data, out[1:].ctypes.data)
        count, first = int(out[0]), int(out[1])
        return count, (None if first == 2**64 - 1 else first)

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())


# Block formats of the typed functions (the same numbering as the library's gq_type).
TYPE_Q4_0, TYPE_Q4_1, TYPE_Q8_0, TYPE_Q4_K, TYPE_Q5_0, TYPE_Q5_1 = 0, 1, 2, 3, 4, 5
BLOCK_BYTES = {TYPE_Q4_0: 18, TYPE_Q4_1: 20, TYPE_Q8_0: 34, TYPE_Q4_K: 144, TYPE_Q5_0: 22, TYPE_Q5_1: 24}
BLOCK_WEIGHTS = {TYPE_Q4_0: 32, TYPE_Q4_1: 32, TYPE_Q8_0: 32, TYPE_Q4_K: 256, TYPE_Q5_0: 32, TYPE_Q5_1: 32}


def get() -> Oracle:
    """The oracle built from this directory's source (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            if _stale(LIB_PATH):
                build_library()
            _lib = Oracle(LIB_PATH)
        return _lib


def within_tolerance(y, y_ref, s_ref, rel: float = 1e-3, abs_: float = 1e-5):
    """MUL_MAT acceptance: |y - y_ref| <= rel * sum_k |w_k x_k| + abs, per element.

    Returns (ok, worst_ratio) where ratio = |y - y_ref| / (rel*s_ref + abs).
    """
    y = np.asarray(y, dtype=np.float64)
    bound = rel * np.asarray(s_ref, dtype=np.float64) + abs_
    err = np.abs(y - np.asarray(y_ref, dtype=np.float64))
    err = np.where(np.isnan(err), np.inf, err)
    ratio = err / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    return bool(worst <= 1.0), worst
