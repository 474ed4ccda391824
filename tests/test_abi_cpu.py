"""The C-ABI library builds, loads and exports every symbol include/gq.h
declares; host-only entry points behave (no GPU needed, no kernel launched)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gq_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    import __graft_entry__
    __graft_entry__._gq_build_module().build()
    import quantized_block_q4_gb300 as gq
    return gq


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("gq_dequant_q4_0", "gq_mul_mat_q4_0", "gq_q4_0_nbytes", "gq_sync_status"):
        assert must in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in gq.h but not exported"
        assert name in lib.SIGNATURES, f"{name} has no Python binding"
        assert hasattr(lib, name), f"{name} missing from the Python module"


def test_host_only_calls(lib):
    assert lib.gq_q4_0_nbytes(11008, 4096) == 11008 * 128 * 18
    assert lib.gq_q4_0_nbytes(1, 33) == 0
    assert lib.gq_q4_0_nbytes(-1, 32) == 0
    assert lib.gq_version() >= 100
    assert lib.gq_status_string(-6) == "GQ_ERR_DEVICE_TIMEOUT"
    old = lib.gq_get_option(lib.GQ_OPT_PREFILL_MIN_N)
    lib.gq_set_option(lib.GQ_OPT_PREFILL_MIN_N, 128)
    assert lib.gq_get_option(lib.GQ_OPT_PREFILL_MIN_N) == 128
    lib.gq_set_option(lib.GQ_OPT_PREFILL_MIN_N, old)
    with pytest.raises(lib.GQError) as e:
        lib.gq_set_option(lib.GQ_OPT_WAIT_LIMIT_NS, 5)
    assert e.value.status == lib.GQ_ERR_SHAPE


def test_argument_errors_before_any_device_work(lib):
    L = lib._lib
    assert L.gq_mul_mat_q4_0(None, 4, 33, None, 1, None, None) == lib.GQ_ERR_SHAPE
    assert "multiple of 32" in lib.gq_last_error()
    assert L.gq_mul_mat_q4_0(None, -4, 32, None, 1, None, None) == lib.GQ_ERR_SHAPE
    assert L.gq_mul_mat_q4_0(None, 1 << 31, 32, None, 1, None, None) == lib.GQ_ERR_SHAPE
    assert L.gq_mul_mat_q4_0(None, 4, 32, None, 1, None, None) == lib.GQ_ERR_NULL
    assert L.gq_mul_mat_q4_0(None, 0, 32, None, 1, None, None) == lib.GQ_OK      # empty
    assert L.gq_mul_mat_q4_0(None, 4, 32, None, 0, None, None) == lib.GQ_OK
    assert L.gq_dequant_q4_0(None, 4, 48, None, None) == lib.GQ_ERR_SHAPE
    assert L.gq_dequant_q4_0(None, 0, 64, None, None) == lib.GQ_OK
    assert L.gq_f32_to_bf16(None, None, -1, None) == lib.GQ_ERR_SHAPE
    L2 = L.gq_mul_mat_id_q4_0
    assert L2(None, 0, 4, 32, None, 2, None, 1, None, None) == lib.GQ_ERR_SHAPE          # n_expert < 1
    assert L2(None, 2, 4, 33, None, 2, None, 1, None, None) == lib.GQ_ERR_SHAPE          # K % 32
    assert L2(None, 2, 4, 32, None, -1, None, 1, None, None) == lib.GQ_ERR_SHAPE         # negative n_ids
    assert L2(None, 2, 4, 32, None, 1 << 20, None, 1 << 12, None, None) == lib.GQ_ERR_SHAPE  # T*n_ids >= 2^31
    assert L2(None, 2, 4, 32, None, 2, None, 0, None, None) == lib.GQ_OK                 # no tokens
    assert L2(None, 2, 0, 32, None, 2, None, 3, None, None) == lib.GQ_OK                 # no rows
    assert L2(None, 2, 4, 32, None, 2, None, 3, None, None) == lib.GQ_ERR_NULL
    assert L.gq_validate(1, None, 4, 33, None, None) == lib.GQ_ERR_SHAPE                # K % 32
    assert L.gq_validate(7, None, 4, 32, None, None) == lib.GQ_ERR_SHAPE                # unknown type
    assert L.gq_validate(0, None, -1, 32, None, None) == lib.GQ_ERR_SHAPE               # negative rows
    assert L.gq_validate(0, None, 4, 32, None, None) == lib.GQ_ERR_NULL                 # no result
    assert L.gq_validate_q4_0(None, 4, 32, 8 * 1024 + 4, None) == lib.GQ_ERR_ALIGN      # result misaligned
    assert L.gq_validate_q4_0(None, 4, 32, 8 * 1024, None) == lib.GQ_ERR_NULL           # W NULL, M*K > 0
    # the repack: a prepared row of K = 2^32 weights would exceed 2^31 bytes (no
    # device access: the pointers are never dereferenced)
    assert L.gq_prepare_q4_0(256, 1, 1 << 32, 0, 256, None) == lib.GQ_ERR_SHAPE
    assert "2^31" in lib.gq_last_error()
    assert L.gq_prepare_q4_0(None, 4, 48, 0, None, None) == lib.GQ_ERR_SHAPE              # K % 32
    assert lib.gq_status_string(-8) == "GQ_ERR_BAD_INDEX"
    old = lib.gq_get_option(lib.GQ_OPT_MOE_PATH)
    with pytest.raises(lib.GQError):
        lib.gq_set_option(lib.GQ_OPT_MOE_PATH, 3)
    lib.gq_set_option(lib.GQ_OPT_MOE_PATH, 2)
    assert lib.gq_get_option(lib.GQ_OPT_MOE_PATH) == 2
    lib.gq_set_option(lib.GQ_OPT_MOE_PATH, old)


def test_timeout_test_hook_option(lib):
    """GQ_OPT_TEST_DROP_ARRIVE: off by default, takes 0..2 only."""
    assert lib.gq_get_option(lib.GQ_OPT_TEST_DROP_ARRIVE) == 0
    with pytest.raises(lib.GQError):
        lib.gq_set_option(lib.GQ_OPT_TEST_DROP_ARRIVE, 3)
    with pytest.raises(lib.GQError):
        lib.gq_set_option(lib.GQ_OPT_TEST_DROP_ARRIVE, -1)
    for v in (1, 2, 0):
        lib.gq_set_option(lib.GQ_OPT_TEST_DROP_ARRIVE, v)
        assert lib.gq_get_option(lib.GQ_OPT_TEST_DROP_ARRIVE) == v
