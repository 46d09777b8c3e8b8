"""The C-ABI library builds, loads without a GPU, exports every function that
include/fd.h declares, and rejects bad arguments on the host before any CUDA
call is made (so these run on a machine without a GPU)."""
import ctypes

import pytest

import long_context_decode_split_gb300 as fd
from long_context_decode_split_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fd.load()


def test_exports_every_declared_symbol(lib):
    declared = fd.header_symbols()
    assert len(declared) >= 10
    for name in declared:
        assert hasattr(lib, name), name
    for name in ("fd_decode_dense", "fd_decode_paged", "fd_quantize_keys", "fd_decode_topdelta"):
        assert name in declared


def test_version_and_status_strings(lib):
    assert fd.fd_abi_version() == 2
    for code in range(7):
        assert fd.fd_status_string(code).startswith("FD_")
    assert "unknown" in fd.fd_status_string(99)


def test_explicit_split_plan_and_workspace(lib):
    # with an explicit chunk count the plan needs no device query
    assert fd.fd_num_splits(1, 32, 32, 32768, 128, 4) == 4
    assert fd.fd_decode_workspace_size(2, 8, 2, 1000, 64, 1) == 0
    assert fd.fd_decode_workspace_size(2, 8, 2, 1000, 64, 3) == 2 * 8 * 3 * (64 + 2) * 4 + 256


P = ctypes.c_void_p


def dense(lib, d=128, Hq=8, Hkv=2, splits=2, ptr=0x10000, ws=None, wsb=0, out_dtype=1):
    a = P(ptr)
    return lib.fd_decode_dense(a, a, a, None, 1, Hq, Hkv, 256, d, 0.1, splits, a, out_dtype, None,
                               ws, wsb, None)


def test_host_validation_codes(lib):
    assert dense(lib, d=96) == fd.FD_ERR_UNSUPPORTED
    assert dense(lib, Hq=18, Hkv=2) == fd.FD_ERR_UNSUPPORTED          # group of 9
    assert dense(lib, Hq=7, Hkv=2) == fd.FD_ERR_INVALID_ARG           # not divisible
    assert dense(lib, splits=-1) == fd.FD_ERR_INVALID_ARG
    assert dense(lib, ptr=0x10008) == fd.FD_ERR_INVALID_ARG           # not 16-byte aligned
    assert dense(lib, out_dtype=7) == fd.FD_ERR_INVALID_ARG
    assert dense(lib, splits=2, ws=None, wsb=0) == fd.FD_ERR_WORKSPACE_TOO_SMALL
    a = P(0x10000)
    # page size other than 64 is not supported; a missing page table is invalid
    assert lib.fd_decode_paged(a, a, a, a, 4, 4, a, 32, 1, 8, 2, 128, 0.1, 1, a, 1, None, None, 0,
                               None) == fd.FD_ERR_UNSUPPORTED
    assert lib.fd_decode_paged(a, a, a, None, 4, 4, a, 64, 1, 8, 2, 128, 0.1, 1, a, 1, None, None, 0,
                               None) == fd.FD_ERR_INVALID_ARG
    # encoder: d must be 64 or 128
    assert lib.fd_quantize_keys(a, None, 1, 2, 64, 96, a, a, a, a, None) == fd.FD_ERR_UNSUPPORTED
    # top-delta: negative delta or window, NaN delta
    args = [a, a, a, a, a, a, None, 1, 8, 2, 128, 128, 0.1]
    tail = [1, a, 1, None, None, None, None, 0, None]
    assert lib.fd_decode_topdelta(*args, -1.0, 4, 64, *tail) == fd.FD_ERR_INVALID_ARG
    assert lib.fd_decode_topdelta(*args, float("nan"), 4, 64, *tail) == fd.FD_ERR_INVALID_ARG
    assert lib.fd_decode_topdelta(*args, 5.0, 4, -1, *tail) == fd.FD_ERR_INVALID_ARG
    # L_max not a multiple of 4; more cache rows than 32-bit tile coordinates reach
    bad_l = [a, a, a, a, a, a, None, 1, 8, 2, 130, 128, 0.1]
    assert lib.fd_decode_topdelta(*bad_l, 5.0, 4, 64, *tail) == fd.FD_ERR_UNSUPPORTED
    huge = [a, a, a, a, a, a, None, 40000, 8, 8, 1 << 16, 128, 0.1]
    assert lib.fd_decode_topdelta(*huge, 5.0, 4, 64, *tail) == fd.FD_ERR_UNSUPPORTED
    assert lib.fd_decode_dense(a, a, a, None, 40000, 8, 8, 1 << 16, 128, 0.1, 1, a, 1, None, None, 0,
                               None) == fd.FD_ERR_UNSUPPORTED


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError):
        fd.open_library(str(tmp_path / "missing.so"))


def test_fp8_host_validation(lib):
    a = P(0x10000)
    f = ctypes.c_float
    # d other than 64/128, misaligned scales, missing scales, group of 9
    assert lib.fd_decode_dense_fp8(a, a, a, a, a, None, 1, 8, 2, 256, 96, 0.1, 1, a, 1, None, None, 0,
                                   None) == fd.FD_ERR_UNSUPPORTED
    assert lib.fd_decode_dense_fp8(a, a, P(0x10004), a, a, None, 1, 8, 2, 256, 128, 0.1, 1, a, 1, None, None,
                                   0, None) == fd.FD_ERR_INVALID_ARG
    assert lib.fd_decode_dense_fp8(a, a, None, a, a, None, 1, 8, 2, 256, 128, 0.1, 1, a, 1, None, None, 0,
                                   None) == fd.FD_ERR_INVALID_ARG
    assert lib.fd_decode_dense_fp8(a, a, a, a, a, None, 1, 18, 2, 256, 128, 0.1, 1, a, 1, None, None, 0,
                                   None) == fd.FD_ERR_UNSUPPORTED
    assert lib.fd_decode_paged_fp8(a, a, a, a, a, a, 4, 4, a, 32, 1, 8, 2, 128, 0.1, 1, a, 1, None, None, 0,
                                   None) == fd.FD_ERR_UNSUPPORTED
    assert lib.fd_quantize_kv_fp8(a, None, 1, 2, 100, 128, a, P(0x10008), None) == fd.FD_ERR_INVALID_ARG
    assert lib.fd_quantize_kv_fp8(a, None, 1, 2, 100, 80, a, a, None) == fd.FD_ERR_UNSUPPORTED
    assert fd.fd_num_splits_fp8(1, 32, 32, 32768, 128, 6) == 6
    assert fd.fd_decode_fp8_workspace_size(2, 8, 2, 1000, 64, 3) == 2 * 8 * 3 * (64 + 2) * 4 + 256


def test_fp4_host_validation(lib):
    a = P(0x10000)
    assert lib.fd_decode_dense_fp4(a, a, a, a, a, None, 1, 8, 2, 256, 96, 0.1, 1, a, 1, None, None, 0,
                                   None) == fd.FD_ERR_UNSUPPORTED
    assert lib.fd_decode_dense_fp4(a, a, P(0x10004), a, a, None, 1, 8, 2, 256, 128, 0.1, 1, a, 1, None, None,
                                   0, None) == fd.FD_ERR_INVALID_ARG
    assert lib.fd_decode_dense_fp4(a, a, None, a, a, None, 1, 8, 2, 256, 128, 0.1, 1, a, 1, None, None, 0,
                                   None) == fd.FD_ERR_INVALID_ARG
    assert lib.fd_decode_paged_fp4(a, a, a, a, a, a, 4, 4, a, 32, 1, 8, 2, 128, 0.1, 1, a, 1, None, None, 0,
                                   None) == fd.FD_ERR_UNSUPPORTED
    assert lib.fd_quantize_kv_fp4(a, None, 1, 2, 100, 128, a, P(0x10008), None) == fd.FD_ERR_INVALID_ARG
    assert lib.fd_quantize_v_fp4(a, None, 1, 2, 100, 128, a, P(0x10008), None) == fd.FD_ERR_INVALID_ARG
    assert lib.fd_quantize_v_fp4(a, None, 1, 2, 100, 96, a, a, None) == fd.FD_ERR_UNSUPPORTED
    assert fd.fd_num_splits_fp4(1, 32, 32, 32768, 128, 6) == 6
    assert fd.fd_decode_fp4_workspace_size(2, 8, 2, 1000, 64, 3) == 2 * 8 * 3 * (64 + 2) * 4 + 256


def test_unified_max_host_validation(lib):
    a = P(0x10000)
    for phi in (float("inf"), float("nan"), 1e31):
        assert lib.fd_decode_dense_unified(a, a, a, None, 1, 8, 2, 256, 128, 0.1, phi, 1, a, 1, None, None, 0,
                                           None) == fd.FD_ERR_INVALID_ARG
        assert lib.fd_decode_paged_unified(a, a, a, a, 4, 4, a, 64, 1, 8, 2, 128, 0.1, phi, 1, a, 1, None,
                                           None, 0, None) == fd.FD_ERR_INVALID_ARG
    # the other checks are fd_decode_dense's
    assert lib.fd_decode_dense_unified(a, a, a, None, 1, 8, 2, 256, 96, 0.1, 6.5, 1, a, 1, None, None, 0,
                                       None) == fd.FD_ERR_UNSUPPORTED
    assert lib.fd_decode_dense_unified(a, a, a, None, 1, 8, 2, 256, 128, 0.1, 6.5, 2, a, 1, None, None, 0,
                                       None) == fd.FD_ERR_WORKSPACE_TOO_SMALL
