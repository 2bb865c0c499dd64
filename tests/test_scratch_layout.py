"""CPU check of the call-scratch layout: the size the library reserves for a
call's scratch (`upsert_scratch_bytes`) equals the extent the carving of that
scratch into arrays uses (`carve_upsert_scratch`), and the carved arrays are
256-byte aligned, disjoint and inside it, for single mode, dual mode and
assign, with and without the LFU arrays.  The allocation-free
insert_or_assign refuses a batch by the first number and writes by the
second, so the two must agree.  Both are host functions of libhkv.so (pure
pointer arithmetic on a base address); no GPU is used."""
import ctypes

import pytest

from tests.test_abi import lib  # noqa: F401  (module fixture: builds and loads libhkv.so)

KINDS = {"single": 0, "dual": 1, "assign": 2}  # hkv::ScratchKind, in declaration order
BASE = 1 << 40


class UpsertScratch(ctypes.Structure):
    """Field for field the host struct hkv::UpsertScratch."""
    _fields_ = [
        ("map_keys", ctypes.c_uint64), ("map_idx", ctypes.c_uint64),
        ("map_size", ctypes.c_uint32), ("area_shift", ctypes.c_int32),
        ("cursor", ctypes.c_uint64), ("mark", ctypes.c_uint64), ("absent", ctypes.c_uint64),
        ("retry", ctypes.c_uint64), ("inc", ctypes.c_uint64),
        ("stage_keys", ctypes.c_uint64), ("stage_idx", ctypes.c_uint64),
        ("stage_bkt", ctypes.c_uint64), ("stage_inc", ctypes.c_uint64),
        ("bytes", ctypes.c_size_t),
    ]


@pytest.fixture(scope="module")
def fns(lib):  # noqa: F811
    size = getattr(lib, "_ZN3hkv20upsert_scratch_bytesEmmNS_11ScratchKindEb")
    size.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int, ctypes.c_bool]
    size.restype = ctypes.c_size_t
    carve = getattr(lib, "_ZN3hkv20carve_upsert_scratchEPvmmNS_11ScratchKindEb")
    carve.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int,
                      ctypes.c_bool]
    carve.restype = UpsertScratch
    return size, carve


def _arrays(s, n, buckets, kind, lfu):
    """(name, start, length in bytes) of every array the carving hands out,
    from the struct's documented meaning of each field."""
    m = s.map_size
    out = [("map_keys", s.map_keys, 8 * m), ("map_idx", s.map_idx, 4 * m), ("cursor", s.cursor, 64)]
    if lfu:
        out.append(("inc", s.inc, 8 * m))
    if kind == "dual":
        out += [("absent", s.absent, m), ("retry", s.retry, 4 * n),
                ("stage_keys", s.stage_keys, 8 * m), ("stage_idx", s.stage_idx, 4 * m),
                ("stage_bkt", s.stage_bkt, 4 * m), ("mark", s.mark, buckets)]
        if lfu:
            out.append(("stage_inc", s.stage_inc, 8 * m))
    elif kind == "single" and s.mark:
        out.append(("mark", s.mark, buckets))
    return out


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("lfu", [False, True])
@pytest.mark.parametrize("n,buckets", [(1, 1), (31, 3), (1000, 512), (4096, 1024), (4097, 1024),
                                       (1 << 20, 1 << 15), (1 << 20, (1 << 23) - 256),
                                       (1 << 19, 12 * (1 << 20) - 256), (3 << 18, 300000)])
def test_carve_matches_reserved_size(fns, kind, lfu, n, buckets):
    size, carve = fns
    want = size(n, buckets, KINDS[kind], lfu)
    s = carve(ctypes.c_void_p(BASE), n, buckets, KINDS[kind], lfu)
    assert s.bytes == want
    assert s.map_size >= 2 * n and s.map_size & (s.map_size - 1) == 0
    spans = sorted((start, start + length, name) for name, start, length in
                   _arrays(s, n, buckets, kind, lfu))
    for lo, hi, name in spans:
        assert lo % 256 == 0, name
        assert BASE <= lo and hi <= BASE + want, name
    for (_, hi, a), (lo, _, b) in zip(spans, spans[1:]):
        assert hi <= lo, (a, b)
    if kind == "single":
        # the single-mode stage is the dedup map itself; marks only for
        # sparse batches (at most 4 keys per bucket)
        assert s.stage_keys == s.map_keys and s.stage_idx == s.map_idx
        assert bool(s.mark) == (n <= 4 * buckets)


def _a(x):
    return (x + 255) // 256 * 256


def _header_bytes(n, buckets, kind, lfu):
    """The allocation-free call's scratch size as include/hkv.h states it."""
    m = 64
    while m < max(64, 2 * n):
        m *= 2
    if kind == "single":
        b = _a(8 * m) + _a(4 * m) + 256 + _a(buckets)
    else:
        b = 2 * _a(8 * m) + 3 * _a(4 * m) + _a(m) + 256 + _a(4 * n) + _a(buckets)
    if lfu:
        b += _a(8 * m) * (2 if kind == "dual" else 1)
    return b


@pytest.mark.parametrize("kind", ["single", "dual"])
@pytest.mark.parametrize("lfu", [False, True])
@pytest.mark.parametrize("n,buckets", [(1, 1), (1000, 512), (1 << 19, 777), (1 << 20, 1 << 15)])
def test_header_formula_is_the_reserved_size(fns, kind, lfu, n, buckets):
    size, _ = fns
    assert size(n, buckets, KINDS[kind], lfu) == _header_bytes(n, buckets, kind, lfu)


def test_noalloc_limits_stated_in_the_header(fns):
    """Single mode: 2^20 keys fit for at most 2^23 - 256 buckets, 2^19 keys
    under LFU for at most 12 * 2^20 - 256; one key more never fits."""
    size, _ = fns
    cap = 32 << 20  # HKV_NOALLOC_SCRATCH_BYTES
    one = KINDS["single"]
    assert size(1 << 20, (1 << 23) - 256, one, False) <= cap
    assert size(1 << 20, (1 << 23) - 255, one, False) > cap
    assert size(1 << 19, 12 * (1 << 20) - 256, one, True) <= cap
    assert size(1 << 19, 12 * (1 << 20) - 255, one, True) > cap
    assert size((1 << 20) + 1, 1, one, False) > cap
    assert size((1 << 19) + 1, 1, one, True) > cap
