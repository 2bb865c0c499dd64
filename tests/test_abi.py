"""CPU checks of the C-ABI library: it builds for sm_103a, loads without a GPU
and exports every function include/hkv.h declares.  No compute calls."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "hkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hkv_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from hash_table_cache_gb300 import _build
    import hash_table_cache_gb300 as hkv
    _build.build()
    return hkv.load()


def test_header_declares_the_abi():
    names = _declared()
    for must in ("hkv_create", "hkv_find", "hkv_insert_or_assign", "hkv_assign", "hkv_erase",
                 "hkv_size", "hkv_export"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_lists_every_declared_symbol():
    import hash_table_cache_gb300 as hkv
    assert sorted(hkv.EXPORTS) == _declared()


def test_status_strings(lib):
    import hash_table_cache_gb300 as hkv
    assert hkv.hkv_status_string(0) == "ok"
    assert "invalid" in hkv.hkv_status_string(-1)


def test_built_for_sm103a_only(lib):
    """The library carries sm_103a code (checked by the build flags)."""
    from hash_table_cache_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_invalid_arguments_rejected_without_gpu(lib):
    """Argument checks run before any CUDA call."""
    import ctypes
    import hash_table_cache_gb300 as hkv
    h = ctypes.c_void_p()
    assert lib.hkv_create(100, 8, 0, 0, 0, ctypes.byref(h)) == hkv.HKV_ERR_INVALID  # not % 128
    assert lib.hkv_create(128, 0, 0, 0, 0, ctypes.byref(h)) == hkv.HKV_ERR_INVALID  # dim 0
    assert lib.hkv_create(128, 8, 1, 0, 0, ctypes.byref(h)) == hkv.HKV_ERR_INVALID  # dual, B=1
    assert lib.hkv_create(256, 8, 8, 0, 0, ctypes.byref(h)) == hkv.HKV_ERR_INVALID  # bad mode
    assert lib.hkv_find(None, 1, None, None, None, None, None) == hkv.HKV_ERR_INVALID
    assert lib.hkv_insert_or_assign(None, 1, None, None, None, None) == hkv.HKV_ERR_INVALID
