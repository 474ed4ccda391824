"""Python binding of the gq C ABI (``include/gq.h``): Q4_0 MUL_MAT on GB300.

Argument marshalling only: every step of dequantisation and MUL_MAT runs in the
CUDA kernels of ``libgq.so``.  PyTorch is used for device memory and streams.
The functions named ``gq_*`` mirror the C entry points one to one and take
torch CUDA tensors (or raw device addresses as ints); ``dequant_q4_0`` and
``mul_mat_q4_0`` / ``mul_mat_id_q4_0`` are conveniences that allocate their outputs with torch.

If ``libgq.so`` is missing this module refuses to import: there is no CPU or
PyTorch fallback.  Build it with ``python quantized_block_q4_gb300/build.py``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgq.so")

GQ_OK = 0
GQ_ERR_NULL = -1
GQ_ERR_SHAPE = -2
GQ_ERR_ALIGN = -3
GQ_ERR_CUDA = -4
GQ_ERR_ALLOC = -5
GQ_ERR_DEVICE_TIMEOUT = -6
GQ_ERR_UNSUPPORTED = -7
GQ_ERR_BAD_INDEX = -8

GQ_TYPE_Q4_0, GQ_TYPE_Q4_1, GQ_TYPE_Q8_0, GQ_TYPE_Q4_K, GQ_TYPE_Q5_0, GQ_TYPE_Q5_1 = 0, 1, 2, 3, 4, 5
TYPE_BLOCK_BYTES = {GQ_TYPE_Q4_0: 18, GQ_TYPE_Q4_1: 20, GQ_TYPE_Q8_0: 34, GQ_TYPE_Q4_K: 144, GQ_TYPE_Q5_0: 22,
                    GQ_TYPE_Q5_1: 24}
TYPE_BLOCK_WEIGHTS = {GQ_TYPE_Q4_0: 32, GQ_TYPE_Q4_1: 32, GQ_TYPE_Q8_0: 32, GQ_TYPE_Q4_K: 256, GQ_TYPE_Q5_0: 32,
                      GQ_TYPE_Q5_1: 32}

GQ_OPT_PREFILL_MIN_N = 0
GQ_OPT_FORCE_GENERIC = 1
GQ_OPT_WAIT_LIMIT_NS = 2
GQ_OPT_WEIGHTS_STATIC = 3
GQ_OPT_DECODE_VARIANT = 4
GQ_OPT_PDL = 5
GQ_OPT_PREFILL_TILE_N = 6
GQ_OPT_PREFILL_PAIR = 7
GQ_OPT_PREFILL_STREAMK = 8
GQ_OPT_PREFILL_SLOTS = 9
GQ_OPT_DECODE_EARLY_STAGES = 10
GQ_OPT_X_STATIC = 11
GQ_OPT_MOE_PATH = 12
GQ_OPT_TEST_DROP_ARRIVE = 13

# Every symbol include/gq.h declares, with (restype, argtypes).
_i64, _sz, _vp, _i32 = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
SIGNATURES = {
    "gq_q4_0_nbytes": (_sz, [_i64, _i64]),
    "gq_dequant_q4_0": (_i32, [_vp, _i64, _i64, _vp, _vp]),
    "gq_type_nbytes": (_sz, [_i32, _i64, _i64]),
    "gq_dequant": (_i32, [_i32, _vp, _i64, _i64, _vp, _vp]),
    "gq_validate": (_i32, [_i32, _vp, _i64, _i64, _vp, _vp]),
    "gq_validate_q4_0": (_i32, [_vp, _i64, _i64, _vp, _vp]),
    "gq_mul_mat": (_i32, [_i32, _vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "gq_quantize_q4_0": (_i32, [_vp, _i64, _i64, _vp, _vp]),
    "gq_mul_mat_q4_0": (_i32, [_vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "gq_prepared_q4_0_nbytes": (_sz, [_i64, _i64]),
    "gq_prepare_q4_0": (_i32, [_vp, _i64, _i64, _i64, _vp, _vp]),
    "gq_mul_mat_q4_0_prepared": (_i32, [_vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "gq_mul_mat_id_q4_0": (_i32, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp]),
    "gq_mul_mat_q4_0_bf16x": (_i32, [_vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "gq_mul_mat_q4_0_noalloc": (_i32, [_vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "gq_f32_to_bf16": (_i32, [_vp, _vp, _i64, _vp]),
    "gq_sync_status": (_i32, [_vp]),
    "gq_set_option": (_i32, [_i32, _i64]),
    "gq_get_option": (_i64, [_i32]),
    "gq_last_error": (ctypes.c_char_p, []),
    "gq_status_string": (ctypes.c_char_p, [_i32]),
    "gq_version": (_i32, []),
}


class GQError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python quantized_block_q4_gb300/build.py` "
                          "(there is no fallback implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _check(status: int) -> None:
    if status != GQ_OK:
        name = _lib.gq_status_string(status).decode()
        raise GQError(status, f"{name}: {_lib.gq_last_error().decode()}")


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor or a device address")
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# ---------------------------------------------------------------- C mirrors
def gq_q4_0_nbytes(M: int, K: int) -> int:
    return int(_lib.gq_q4_0_nbytes(M, K))


def gq_dequant_q4_0(W, M: int, K: int, out, stream=None) -> None:
    _check(_lib.gq_dequant_q4_0(_ptr(W), M, K, _ptr(out), _stream(stream)))


def gq_type_nbytes(qtype: int, M: int, K: int) -> int:
    return int(_lib.gq_type_nbytes(qtype, M, K))


def gq_dequant(qtype: int, W, M: int, K: int, out, stream=None) -> None:
    _check(_lib.gq_dequant(qtype, _ptr(W), M, K, _ptr(out), _stream(stream)))


def gq_validate(qtype: int, W, M: int, K: int, result, stream=None) -> None:
    _check(_lib.gq_validate(qtype, _ptr(W), M, K, _ptr(result), _stream(stream)))


def gq_validate_q4_0(W, M: int, K: int, result, stream=None) -> None:
    _check(_lib.gq_validate_q4_0(_ptr(W), M, K, _ptr(result), _stream(stream)))


def gq_mul_mat(qtype: int, W, M: int, K: int, X, N: int, Y, stream=None) -> None:
    _check(_lib.gq_mul_mat(qtype, _ptr(W), M, K, _ptr(X), N, _ptr(Y), _stream(stream)))


def gq_quantize_q4_0(W, M: int, K: int, out, stream=None) -> None:
    _check(_lib.gq_quantize_q4_0(_ptr(W), M, K, _ptr(out), _stream(stream)))


def gq_mul_mat_q4_0(W, M: int, K: int, X, N: int, Y, stream=None) -> None:
    _check(_lib.gq_mul_mat_q4_0(_ptr(W), M, K, _ptr(X), N, _ptr(Y), _stream(stream)))


def gq_prepared_q4_0_nbytes(M: int, K: int) -> int:
    return int(_lib.gq_prepared_q4_0_nbytes(M, K))


def gq_prepare_q4_0(W, M: int, K: int, row_stride: int, out, stream=None) -> None:
    _check(_lib.gq_prepare_q4_0(_ptr(W), M, K, row_stride, _ptr(out), _stream(stream)))


def gq_mul_mat_q4_0_prepared(Wp, M: int, K: int, X, N: int, Y, stream=None) -> None:
    _check(_lib.gq_mul_mat_q4_0_prepared(_ptr(Wp), M, K, _ptr(X), N, _ptr(Y), _stream(stream)))


def gq_mul_mat_id_q4_0(W, n_expert: int, M: int, K: int, X, n_ids: int, ids, T: int, Y, stream=None) -> None:
    _check(_lib.gq_mul_mat_id_q4_0(_ptr(W), n_expert, M, K, _ptr(X), n_ids, _ptr(ids), T, _ptr(Y),
                                   _stream(stream)))


def gq_mul_mat_q4_0_bf16x(W, M: int, K: int, X_bf16, N: int, Y, stream=None) -> None:
    _check(_lib.gq_mul_mat_q4_0_bf16x(_ptr(W), M, K, _ptr(X_bf16), N, _ptr(Y), _stream(stream)))


def gq_mul_mat_q4_0_noalloc(W, M: int, K: int, X, N: int, Y, stream=None) -> None:
    """Tensor-core MUL_MAT that allocates no device memory (fixed in-library
    scratch); for callers whose memory must come only from their own pool."""
    _check(_lib.gq_mul_mat_q4_0_noalloc(_ptr(W), M, K, _ptr(X), N, _ptr(Y), _stream(stream)))


def gq_f32_to_bf16(x, y, n: int, stream=None) -> None:
    _check(_lib.gq_f32_to_bf16(_ptr(x), _ptr(y), n, _stream(stream)))


def gq_sync_status(stream=None) -> None:
    _check(_lib.gq_sync_status(_stream(stream)))


def gq_set_option(opt: int, value: int) -> None:
    _check(_lib.gq_set_option(opt, value))


def gq_get_option(opt: int) -> int:
    return int(_lib.gq_get_option(opt))


def gq_last_error() -> str:
    return _lib.gq_last_error().decode()


def gq_status_string(status: int) -> str:
    return _lib.gq_status_string(status).decode()


def gq_version() -> int:
    return int(_lib.gq_version())


# ---------------------------------------------------------------- conveniences
def _check_w(W: torch.Tensor, K: int) -> int:
    if W.dtype != torch.uint8:
        raise TypeError("W must be uint8 (raw block_q4_0 bytes)")
    if K % 32 or K <= 0:
        raise ValueError("K must be a positive multiple of 32")
    row = K // 32 * 18
    if W.numel() % row:
        raise ValueError("W size is not a whole number of rows")
    return W.numel() // row


def dequant_q4_0(W: torch.Tensor, K: int, stream=None) -> torch.Tensor:
    """W: uint8 [M, K/32*18] -> float32 [M, K] (bit-exact d*(q-8))."""
    M = _check_w(W, K)
    out = torch.empty((M, K), dtype=torch.float32, device=W.device)
    gq_dequant_q4_0(W, M, K, out, stream)
    return out


def quantize_q4_0(W: torch.Tensor, stream=None) -> torch.Tensor:
    """W: float32 [M, K] (K % 32 == 0) -> uint8 [M, K/32*18] Q4_0 blocks."""
    if W.dtype != torch.float32 or W.dim() != 2 or not W.is_contiguous():
        raise TypeError("W must be a contiguous float32 [M, K] tensor")
    M, K = W.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    out = torch.empty((M, K // 32 * 18), dtype=torch.uint8, device=W.device)
    gq_quantize_q4_0(W, M, K, out, stream)
    return out


def mul_mat_q4_0(W: torch.Tensor, X: torch.Tensor, stream=None, out: torch.Tensor | None = None) -> torch.Tensor:
    """Y[N, M] = X[N, K] @ dequant(W)^T with W uint8 [M, K/32*18], X float32 [N, K]."""
    if X.dtype != torch.float32 or X.dim() != 2:
        raise TypeError("X must be float32 [N, K]")
    N, K = X.shape
    M = _check_w(W, K)
    Y = out if out is not None else torch.empty((N, M), dtype=torch.float32, device=X.device)
    gq_mul_mat_q4_0(W, M, K, X, N, Y, stream)
    return Y


def mul_mat_id_q4_0(W: torch.Tensor, n_expert: int, X: torch.Tensor, ids: torch.Tensor, stream=None,
                    out: torch.Tensor | None = None) -> torch.Tensor:
    """Y[T, S, M]: row (t, s) is X[t, s] @ dequant(W_e)^T with e = ids[t, s].
    W uint8 [n_expert*M, K/32*18] (experts one after the other), X float32
    [T, S, K], ids int32 [T, S]."""
    if X.dtype != torch.float32 or X.dim() != 3:
        raise TypeError("X must be float32 [T, S, K]")
    if ids.dtype != torch.int32 or tuple(ids.shape) != tuple(X.shape[:2]):
        raise TypeError("ids must be int32 [T, S]")
    T, S, K = X.shape
    rows = _check_w(W, K)
    if n_expert < 1 or rows % n_expert:
        raise ValueError("W rows are not a multiple of n_expert")
    M = rows // n_expert
    Y = out if out is not None else torch.empty((T, S, M), dtype=torch.float32, device=X.device)
    gq_mul_mat_id_q4_0(W, n_expert, M, K, X, S, ids, T, Y, stream)
    return Y


def _rows_of(W: torch.Tensor, qtype: int, K: int) -> int:
    if W.dtype != torch.uint8:
        raise TypeError("W must be uint8 (raw blocks)")
    bw = TYPE_BLOCK_WEIGHTS[qtype]
    if K % bw or K <= 0:
        raise ValueError(f"K must be a positive multiple of {bw}")
    row = K // bw * TYPE_BLOCK_BYTES[qtype]
    if W.numel() % row:
        raise ValueError("W size is not a whole number of rows")
    return W.numel() // row


def dequant(qtype: int, W: torch.Tensor, K: int, stream=None) -> torch.Tensor:
    """W: uint8 rows of blocks of type qtype -> float32 [M, K] (bit-exact)."""
    M = _rows_of(W, qtype, K)
    out = torch.empty((M, K), dtype=torch.float32, device=W.device)
    gq_dequant(qtype, W, M, K, out, stream)
    return out


def validate(qtype: int, W: torch.Tensor, K: int, M: int | None = None, stream=None):
    """Blocks of W (block format qtype) with a NaN or infinite scale field:
    (count, first flat block index or None).  Synchronises the stream."""
    if W.dtype != torch.uint8:
        raise TypeError("W must be uint8 (raw block bytes)")
    if M is None:
        M = _rows_of(W, qtype, K)
    result = torch.empty(2, dtype=torch.int64, device=W.device)
    gq_validate(qtype, W, M, K, result, stream)
    if stream is not None:
        stream.synchronize()
    r = result.cpu().tolist()  # uint64 values read as int64: mask back to unsigned
    count, first = int(r[0]), int(r[1]) & 0xFFFFFFFFFFFFFFFF
    return count, (None if first == 0xFFFFFFFFFFFFFFFF else first)


def mul_mat(qtype: int, W: torch.Tensor, X: torch.Tensor, stream=None, out: torch.Tensor | None = None) -> torch.Tensor:
    """Y[N, M] = X[N, K] @ dequant(W)^T for W in block format qtype."""
    if X.dtype != torch.float32 or X.dim() != 2:
        raise TypeError("X must be float32 [N, K]")
    N, K = X.shape
    M = _rows_of(W, qtype, K)
    Y = out if out is not None else torch.empty((N, M), dtype=torch.float32, device=X.device)
    gq_mul_mat(qtype, W, M, K, X, N, Y, stream)
    return Y


def prepare_q4_0(W: torch.Tensor, K: int, row_stride: int = 0, M: int | None = None, stream=None) -> torch.Tensor:
    """Q4_0 rows (packed, or row_stride bytes apart) -> the prepared layout
    (uint8 [M, ceil(K/256)*144])."""
    if W.dtype != torch.uint8:
        raise TypeError("W must be uint8 (raw block_q4_0 bytes)")
    if M is None:
        M = _check_w(W, K) if row_stride == 0 else W.numel() // row_stride
    out = torch.empty((M, gq_prepared_q4_0_nbytes(1, K)), dtype=torch.uint8, device=W.device)
    gq_prepare_q4_0(W, M, K, row_stride, out, stream)
    return out


def mul_mat_q4_0_prepared(Wp: torch.Tensor, X: torch.Tensor, stream=None) -> torch.Tensor:
    """Y[N, M] = X[N, K] @ dequant(W)^T with Wp = prepare_q4_0(W, K)."""
    N, K = X.shape
    M = Wp.shape[0]
    Y = torch.empty((N, M), dtype=torch.float32, device=X.device)
    gq_mul_mat_q4_0_prepared(Wp, M, K, X, N, Y, stream)
    return Y
