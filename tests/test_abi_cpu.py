"""CPU-only checks of the C ABI: the library builds, loads, exports every
symbol include/mla.h declares, and rejects bad arguments on the host before
touching the GPU."""
import ctypes
import os
import re

import pytest

import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import build as mla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mla_build.build()
    return mla.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(mla_\w+)\s*\(", text, flags=re.M)))


def test_header_symbols_exported(lib):
    declared = _declared_functions()
    assert len(declared) >= 10, declared
    assert set(declared) == set(mla.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert mla.version() >= 100
    assert mla.status_string(0) == "ok"
    for s in range(-6, 0):
        assert mla.status_string(s) != "unknown status"


def test_check_dims(lib):
    assert mla.check_dims(mla.dims(16, 64)) == mla.MLA_OK
    assert mla.check_dims(mla.dims(128, 16, int8=True)) == mla.MLA_OK
    assert mla.check_dims(mla.dims(16, 64, fp8=True)) == mla.MLA_OK
    assert mla.check_dims(mla.dims(128, 128, fp8=True)) == mla.MLA_OK
    assert mla.check_dims(mla.dims(64, 32)) == mla.MLA_OK
    assert mla.check_dims(mla.dims(24, 64)) == mla.MLA_ERR_UNSUPPORTED
    assert mla.check_dims(mla.dims(16, 48)) == mla.MLA_ERR_UNSUPPORTED
    assert mla.check_dims(mla.dims(16, 64, kv_lora_rank=256)) == mla.MLA_ERR_UNSUPPORTED
    assert mla.check_dims(mla.dims(0, 64)) == mla.MLA_ERR_INVALID_ARG
    d = mla.dims(16, 64)
    d.cache_dtype = 7
    assert mla.check_dims(d) == mla.MLA_ERR_INVALID_ARG
    d.cache_dtype = 3
    assert mla.check_dims(d) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_check_dims(None) == mla.MLA_ERR_INVALID_ARG


def test_workspace_size_explicit_splits(lib):
    d = mla.dims(16, 64)
    small = lib.mla_decode_workspace_size(ctypes.byref(d), 1, 4)
    big = lib.mla_decode_workspace_size(ctypes.byref(d), 32, 152)
    assert 0 < small < big
    # partials dominate: (splits + batch) * H * 512 fp32
    assert big >= (152 + 32) * 16 * 512 * 4
    assert lib.mla_decode_workspace_size(ctypes.byref(d), 0, 4) == 0
    assert lib.mla_decode_workspace_size(ctypes.byref(d), 4, -1) == 0


def test_host_validation_rejects_before_launch(lib):
    d = mla.dims(16, 64)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    args = [ctypes.byref(d), fake, fake, fake, None, 4, fake, 8, fake, 2, fake, fake, ctypes.c_float(0.1), 4,
            fake, ctypes.c_size_t(1 << 30), fake, None, None]
    a = list(args); a[1] = None                       # q_nope missing
    assert lib.mla_decode(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[9] = 0                          # batch 0
    assert lib.mla_decode(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[12] = ctypes.c_float(-1.0)      # negative scale
    assert lib.mla_decode(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[3] = ctypes.c_void_p(0x10008)   # cache not 16-byte aligned
    assert lib.mla_decode(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[14] = ctypes.c_void_p(0x10040)  # workspace not 256-byte aligned
    assert lib.mla_decode(*a) == mla.MLA_ERR_WORKSPACE
    a = list(args); a[15] = ctypes.c_size_t(16)       # workspace too small
    assert lib.mla_decode(*a) == mla.MLA_ERR_WORKSPACE
    di = mla.dims(16, 64, int8=True)
    a = list(args); a[0] = ctypes.byref(di)           # INT8 without scale/zero array
    assert lib.mla_decode(*a) == mla.MLA_ERR_INVALID_ARG
    df = mla.dims(16, 64, fp8=True)
    a = list(args); a[0] = ctypes.byref(df)           # FP8 without its scales
    assert lib.mla_decode(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[0] = ctypes.byref(df); a[4] = ctypes.c_void_p(0x10004)  # scales not 16-byte aligned
    assert lib.mla_decode(*a) == mla.MLA_ERR_INVALID_ARG
    # append
    assert lib.mla_cache_append(ctypes.byref(d), None, None, 4, fake, 2, 8, fake, fake, 3, fake, fake,
                                ctypes.c_double(1e4), None, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_cache_append(ctypes.byref(d), fake, None, 4, fake, 2, 8, fake, fake, 0, fake, fake,
                                ctypes.c_double(1e4), None, None) == mla.MLA_OK  # no tokens: no-op
    assert lib.mla_cache_append(ctypes.byref(di), fake, None, 4, fake, 2, 8, fake, fake, 3, fake, fake,
                                ctypes.c_double(1e4), None, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_cache_append(ctypes.byref(df), fake, None, 4, fake, 2, 8, fake, fake, 3, fake, fake,
                                ctypes.c_double(1e4), None, None) == mla.MLA_ERR_INVALID_ARG
    # combine
    assert lib.mla_combine(ctypes.byref(d), fake, fake, 2, 0, fake, None, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_combine(ctypes.byref(d), None, fake, 2, 3, fake, None, None) == mla.MLA_ERR_INVALID_ARG
    # timing hook: both or neither
    assert lib.mla_set_timing_events(fake, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_set_timing_events(None, None) == mla.MLA_OK


def test_no_alloc_host_validation(lib):
    """mla_decode_no_alloc returns what mla_decode returns for bad arguments,
    and refuses shapes larger than its fixed scratch before touching a GPU."""
    d = mla.dims(16, 64)
    fake = ctypes.c_void_p(0x10000)

    def call(dims, batch, splits):
        return lib.mla_decode_no_alloc(ctypes.byref(dims), fake, fake, fake, None, 4, fake, 8, fake, batch, fake,
                                       fake, ctypes.c_float(0.1), splits, fake, None, None, None)

    assert call(d, 0, 4) == mla.MLA_ERR_INVALID_ARG
    assert call(d, 4, -1) == mla.MLA_ERR_INVALID_ARG
    assert call(mla.dims(24, 64), 4, 4) == mla.MLA_ERR_UNSUPPORTED
    assert call(mla.dims(0, 64), 4, 4) == mla.MLA_ERR_INVALID_ARG
    assert call(mla.dims(16, 64), 1 << 23, 4) == mla.MLA_ERR_INVALID_ARG  # beyond the query-row limit
    assert lib.mla_decode_workspace_size(ctypes.byref(d), 4096, 152) > mla.NO_ALLOC_WORKSPACE_BYTES
    assert call(d, 4096, 152) == mla.MLA_ERR_WORKSPACE


def test_multi_token_workspace_and_validation(lib):
    d = mla.dims(16, 64)
    # q_len tokens of H heads need the workspace of a q_len * H-head decode
    for T in (1, 2, 4, 8):
        dT = mla.dims(16 * T, 64)
        got = lib.mla_decode_multi_workspace_size(ctypes.byref(d), 32, T, 76)
        assert got == lib.mla_decode_workspace_size(ctypes.byref(dT), 32, 76) > 0
    assert lib.mla_decode_multi_workspace_size(ctypes.byref(d), 32, 0, 76) == 0
    assert lib.mla_decode_multi_workspace_size(ctypes.byref(d), 32, mla.MAX_Q_LEN + 1, 76) == 0
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    args = [ctypes.byref(d), fake, fake, fake, None, 4, fake, 8, fake, 2, 2, fake, fake, ctypes.c_float(0.1), 4,
            fake, ctypes.c_size_t(1 << 30), fake, None, None]
    for bad_t in (0, -1, mla.MAX_Q_LEN + 1):
        a = list(args); a[10] = bad_t
        assert lib.mla_decode_multi(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[1] = None
    assert lib.mla_decode_multi(*a) == mla.MLA_ERR_INVALID_ARG


def test_prefill_workspace_and_validation(lib):
    d = mla.dims(16, 64)
    # a chunk of T tokens needs the workspace of T-token multi-token decode
    for T in (1, 8, 64, 512):
        dT = mla.dims(16 * T, 64)
        got = lib.mla_prefill_workspace_size(ctypes.byref(d), 4, T, 3)
        assert got == lib.mla_decode_workspace_size(ctypes.byref(dT), 4, 3) > 0
    assert lib.mla_prefill_workspace_size(ctypes.byref(d), 4, 0, 3) == 0
    assert lib.mla_prefill_workspace_size(ctypes.byref(d), 4, mla.MAX_PREFILL_CHUNK + 1, 3) == 0
    assert mla.MAX_PREFILL_CHUNK > mla.MAX_Q_LEN
    # more than 2^26 query rows (batch * chunk * H) are refused
    assert lib.mla_prefill_workspace_size(ctypes.byref(mla.dims(128, 64)), 2048, 2048, 3) == 0
    assert lib.mla_prefill_workspace_size(ctypes.byref(mla.dims(128, 64)), 256, 2048, 3) > 0
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    big = ctypes.c_size_t(1 << 40)
    args = [ctypes.byref(d), fake, None, 4, fake, 8, fake, 2, 64, fake, fake, ctypes.c_double(1e4), fake, fake,
            fake, fake, ctypes.c_float(0.1), 3, fake, big, fake, None, None]
    for bad_chunk in (0, -2, mla.MAX_PREFILL_CHUNK + 1):
        a = list(args); a[8] = bad_chunk
        assert lib.mla_prefill(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[9] = None                       # no new rows
    assert lib.mla_prefill(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[12] = None                      # no queries
    assert lib.mla_prefill(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[9] = ctypes.c_void_p(0x10008)   # rows not 16-byte aligned
    assert lib.mla_prefill(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[18] = ctypes.c_void_p(0x10040)  # workspace not 256-byte aligned
    assert lib.mla_prefill(*a) == mla.MLA_ERR_WORKSPACE
    a = list(args); a[19] = ctypes.c_size_t(64)       # workspace too small
    assert lib.mla_prefill(*a) == mla.MLA_ERR_WORKSPACE
    df = mla.dims(16, 64, fp8=True)
    a = list(args); a[0] = ctypes.byref(df)           # FP8 cache without its scales
    assert lib.mla_prefill(*a) == mla.MLA_ERR_INVALID_ARG


def test_sparse_workspace_and_validation(lib):
    d = mla.dims(16, 64)
    dec = lib.mla_decode_workspace_size(ctypes.byref(d), 32, 76)
    sp = lib.mla_decode_sparse_workspace_size(ctypes.byref(d), 32, 2048, 76)
    assert sp >= dec + 32 * 2048 * 1152   # the decode's workspace plus the gathered rows
    # 1-byte caches gather 576-byte rows plus their scales: 8 (INT8) or 4 (FP8) bytes a row
    di, df = mla.dims(16, 64, int8=True), mla.dims(16, 64, fp8=True)
    deci = lib.mla_decode_workspace_size(ctypes.byref(di), 32, 76)
    spi = lib.mla_decode_sparse_workspace_size(ctypes.byref(di), 32, 2048, 76)
    spf = lib.mla_decode_sparse_workspace_size(ctypes.byref(df), 32, 2048, 76)
    assert spi >= deci + 32 * 2048 * (576 + 8) and spf >= deci + 32 * 2048 * (576 + 4)
    assert spf < spi < sp
    assert lib.mla_decode_sparse_workspace_size(ctypes.byref(d), 32, 0, 76) == 0
    assert lib.mla_decode_sparse_workspace_size(ctypes.byref(d), 32, mla.MAX_TOP_K + 1, 76) == 0
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    args = [ctypes.byref(d), fake, fake, fake, None, 4, fake, 8, fake, 2, fake, 64, fake, fake, ctypes.c_float(0.1),
            4, fake, ctypes.c_size_t(1 << 30), fake, None, None]
    for bad_k in (0, -3, mla.MAX_TOP_K + 1):
        a = list(args); a[11] = bad_k
        assert lib.mla_decode_sparse(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[10] = None                      # no index list
    assert lib.mla_decode_sparse(*a) == mla.MLA_ERR_INVALID_ARG
    a = list(args); a[16] = ctypes.c_void_p(0x10010)  # workspace not 256-byte aligned
    assert lib.mla_decode_sparse(*a) == mla.MLA_ERR_WORKSPACE
