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


def test_null_table_is_refused_on_the_host(lib):
    """Every call taking a table refuses a NULL one with HKV_ERR_INVALID
    before touching CUDA (this machine may have no GPU); destroy(NULL) is a
    no-op; hkv_create refuses a bad shape before allocating anything."""
    import ctypes
    import hash_table_cache_gb300 as hkv
    u64 = ctypes.c_uint64
    out = ctypes.c_void_p()
    calls = {
        "hkv_find": (None, 1, None, None, None, None, None),
        "hkv_insert_or_assign": (None, 1, None, None, None, None),
        "hkv_insert_or_assign_noalloc": (None, 1, None, None, None, None),
        "hkv_assign": (None, 1, None, None, None, None),
        "hkv_insert_and_evict": (None, 1, None, None, None, None, None, None, None, None),
        "hkv_find_or_insert": (None, 1, None, None, None, None, None),
        "hkv_contains": (None, 1, None, None, None),
        "hkv_find_ptr": (None, 1, None, None, None, None, None),
        "hkv_erase": (None, 1, None, None),
        "hkv_size": (None, ctypes.byref(u64()), None),
        "hkv_export": (None, 0, 128, 0, None, None, None, None, None),
        "hkv_get_error_counts": (None, ctypes.byref(u64()), ctypes.byref(u64())),
        "hkv_get_op_counts": (None, ctypes.byref(hkv.OpCounts())),
        "hkv_reset_op_counts": (None,),
        "hkv_get_info": (None, ctypes.byref(hkv.Info())),
        "hkv_set_epoch": (None, 3),
    }
    for name, args in calls.items():
        assert getattr(lib, name)(*args) == hkv.HKV_ERR_INVALID, name
    assert lib.hkv_destroy(None) == hkv.HKV_OK
    for cap, dim, mode in ((100, 4, 0), (0, 4, 0), (128, 0, 0), (128, 4, hkv.HKV_MODE_DUAL)):
        assert lib.hkv_create(cap, dim, mode, 0, 0, ctypes.byref(out)) == hkv.HKV_ERR_INVALID
        assert out.value is None


def test_binding_constants_match_the_header():
    """The binding's numeric constants are the header's."""
    import hash_table_cache_gb300 as hkv
    text = open(os.path.join(ROOT, "include", "hkv.h")).read()
    for name in ("HKV_MAX_BATCH", "HKV_SLOTS_PER_BUCKET"):
        m = re.search(r"#define " + name + r" (0x[0-9A-Fa-f]+|\d+)", text)
        assert m, name
        py = hkv.SLOTS_PER_BUCKET if name == "HKV_SLOTS_PER_BUCKET" else hkv.HKV_MAX_BATCH
        assert int(m.group(1), 0) == py, name
    for name, value in (("HKV_OK", hkv.HKV_OK), ("HKV_ERR_INVALID", hkv.HKV_ERR_INVALID),
                        ("HKV_MODE_DUAL", hkv.HKV_MODE_DUAL), ("HKV_MODE_TIERED", hkv.HKV_MODE_TIERED),
                        ("HKV_POLICY_LFU", hkv.HKV_POLICY_LFU)):
        m = re.search(name + r"\s*=\s*(-?(?:0x[0-9A-Fa-f]+|\d+))", text)
        assert m and int(m.group(1), 0) == value, name
