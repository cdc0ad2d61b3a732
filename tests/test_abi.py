"""CPU checks of the C ABI: the library loads without a GPU, exports every
function the headers under include/ declare, and rejects bad arguments on the host."""
import ctypes
import glob
import os
import re

import pytest

import paged_kv_cache_19_gb300 as kp
from paged_kv_cache_19_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return kp.load_library()


def declared_functions(header=None):
    paths = ([os.path.join(ROOT, "include", header)] if header
             else sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))))
    names = set()
    for path in paths:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_expected_calls():
    names = declared_functions("kv_paged.h")
    for must in ("kv_pool_create", "paged_kv_append", "paged_decode_attention",
                 "paged_decode_attention_split_merge", "paged_merge_attention_states",
                 "paged_decode_step", "paged_attention_multi_query"):
        assert must in names
    assert len(names) >= 12
    bm = declared_functions("kv_block_manager.h")
    for must in ("kv_bm_create", "kv_bm_append_slots", "kv_bm_match_prefix", "kv_copy_blocks"):
        assert must in bm


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert lib.kv_abi_version() == 1
    for code in range(7):
        assert lib.kv_status_string(code)
    assert lib.kv_status_string(99) == b"unknown status"


def test_pool_create_validates_on_the_host(lib):
    h = ctypes.c_void_p(123)
    assert lib.kv_pool_create(0, 16, 8, 128, 0, 0, ctypes.byref(h)) == kp.KV_ERR_INVALID_ARG
    assert h.value is None
    assert lib.kv_pool_create(64, 16, 8, 128, 7, 0, ctypes.byref(h)) == kp.KV_ERR_INVALID_ARG
    assert lib.kv_pool_create(64, 24, 8, 128, 0, 0, ctypes.byref(h)) == kp.KV_ERR_UNSUPPORTED
    assert lib.kv_pool_create(64, 16, 8, 96, 0, 0, ctypes.byref(h)) == kp.KV_ERR_UNSUPPORTED
    assert lib.kv_pool_create(64, 16, 8, 64, 1, 0, ctypes.byref(h)) == kp.KV_ERR_UNSUPPORTED
    assert lib.kv_pool_create(1 << 30, 32, 64, 128, 0, 0, ctypes.byref(h)) == kp.KV_ERR_UNSUPPORTED
    assert lib.kv_pool_create(64, 16, 8, 128, 0, 0, None) == kp.KV_ERR_INVALID_ARG


def test_calls_on_a_null_pool_are_rejected(lib):
    n = ctypes.c_size_t()
    assert lib.paged_decode_workspace_size(None, 1, 8, 4, 0, ctypes.byref(n)) == kp.KV_ERR_INVALID_ARG
    assert lib.paged_kv_append(None, None, None, 1, None, None, None, 1, None, 1, None) == \
        kp.KV_ERR_INVALID_ARG
    assert lib.paged_decode_attention(None, None, 8, None, 4, None, 1, 1.0, 0, None, 0, None, None,
                                      None) == kp.KV_ERR_INVALID_ARG
    assert lib.paged_decode_attention_split_merge(None, None, 8, None, 4, None, 1, 1.0, 0, None, 0,
                                                  None, None, None) == kp.KV_ERR_INVALID_ARG
    assert lib.kv_pool_destroy(None) == kp.KV_OK
    bits = ctypes.c_uint32()
    assert lib.kv_pool_device_errors(None, ctypes.byref(bits), 0) == kp.KV_ERR_INVALID_ARG


def test_merge_attention_states_validates_on_the_host(lib):
    """Bad sizes, missing or misaligned pointers are rejected before any launch (the
    pointers are never dereferenced); no rows is a no-op."""
    bad = kp.KV_ERR_INVALID_ARG
    a16, a4 = 1 << 20, (1 << 20) + 4                  # 16-byte and only 4-byte aligned values
    assert lib.paged_merge_attention_states(a16, a16, 0, 4, 64, a16, None, None) == bad
    assert lib.paged_merge_attention_states(a16, a16, 2, -1, 64, a16, None, None) == bad
    for d in (0, 4, 12, 1032):
        assert lib.paged_merge_attention_states(a16, a16, 2, 4, d, a16, None, None) == bad
    assert lib.paged_merge_attention_states(None, a16, 2, 4, 64, a16, None, None) == bad
    assert lib.paged_merge_attention_states(a16, None, 2, 4, 64, a16, None, None) == bad
    assert lib.paged_merge_attention_states(a16, a16, 2, 4, 64, None, None, None) == bad
    assert lib.paged_merge_attention_states(a4, a16, 2, 4, 64, a16, None, None) == bad
    assert lib.paged_merge_attention_states(a16, a16, 2, 4, 64, a4, None, None) == bad
    assert lib.paged_merge_attention_states(a16, a16, 2, 4, 64, a16, a16 + 2, None) == bad
    assert lib.paged_merge_attention_states(None, None, 2, 0, 64, None, None, None) == kp.KV_OK


def test_pool_create_without_a_gpu_reports_a_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    assert lib.kv_pool_create(64, 16, 8, 128, 0, 0, ctypes.byref(h)) == kp.KV_ERR_CUDA


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(kp, "_lib", None)
    monkeypatch.setattr(kp, "_LIB_PATH", "/nonexistent/libkvpaged.so")
    with pytest.raises(RuntimeError, match="not built"):
        kp.load_library()


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_cache_19_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_decode_stall_hook_validates_on_the_host(lib):
    assert lib.kv_debug_decode_stall(-2, ctypes.c_ulonglong(0)) == kp.KV_ERR_INVALID_ARG
    assert lib.kv_debug_decode_stall(-1, ctypes.c_ulonglong(0)) == kp.KV_OK
