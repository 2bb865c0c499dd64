"""Python binding of the cache-semantic GPU hash table (``include/hkv.h``).

The binding only marshals arguments: every step of every operation runs in
the CUDA kernels of ``libhkv.so`` (built in-tree for sm_103a by
``hash_table_cache_gb300._build``).  There is no CPU fallback: if the library
is missing or cannot be loaded, every call raises.

Two layers:

* ``hkv_create`` / ``hkv_find`` / ``hkv_insert_or_assign`` / ... -- the C ABI
  one to one.  Pointer arguments accept a torch tensor (its ``data_ptr()``),
  an int address or None; ``stream`` accepts a ``torch.cuda.Stream``, a raw
  handle or None (the current torch stream).  They return the status code.
* ``HashTable`` -- the same calls on torch tensors, raising ``HKVError`` on a
  non-zero status and allocating outputs.

Semantics follow "HierarchicalKV: A GPU Hash Table with Cache Semantics for
Continuous Online Embedding Storage" (arXiv 2603.17168v1); see the header for
the exact contract of each call.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libhkv.so")

HKV_MODE_SINGLE = 0
HKV_MODE_DUAL = 1
HKV_MODE_TIERED = 2
# score policies, ORed into the mode (HKV §3.3; Table 8 names)
HKV_POLICY_CUSTOMIZED = 0x00
HKV_POLICY_LRU = 0x10
HKV_POLICY_LFU = 0x20
HKV_POLICY_EPOCH_LRU = 0x30
HKV_POLICY_EPOCH_LFU = 0x40
HKV_POLICY_MASK = 0xF0
HKV_OK = 0
HKV_ERR_INVALID = -1
HKV_ERR_OOM = -2
HKV_ERR_CUDA = -3
HKV_ERR_RESERVED_KEY = -4
HKV_ERR_TIMEOUT = -5
SLOTS_PER_BUCKET = 128
RESERVED_KEY_LO = 0xFFFFFFFFFFFFFFF0
HKV_MAX_BATCH = 0x7FFFFFFF  # largest n a batched call accepts

# Every symbol include/hkv.h declares (checked by the CPU test suite).
EXPORTS = (
    "hkv_create", "hkv_destroy", "hkv_find", "hkv_insert_or_assign", "hkv_assign", "hkv_erase",
    "hkv_size", "hkv_export", "hkv_get_error_counts", "hkv_get_op_counts",
    "hkv_reset_op_counts", "hkv_get_info", "hkv_status_string", "hkv_insert_or_assign_noalloc",
    "hkv_insert_and_evict", "hkv_find_or_insert", "hkv_contains", "hkv_find_ptr",
    "hkv_set_epoch",
)
NOALLOC_SCRATCH_BYTES = 32 << 20


class HKVError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = _lib_or_none().hkv_status_string(status).decode() if _lib_or_none() else str(status)
        super().__init__(f"{what}: {msg} ({status})" if what else f"{msg} ({status})")


class OpCounts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("updated", "admitted", "evicted", "rejected", "erased")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class Info(ctypes.Structure):
    _fields_ = [("capacity", ctypes.c_uint64), ("num_buckets", ctypes.c_uint64),
                ("hbm_value_rows", ctypes.c_uint64), ("dim", ctypes.c_uint32),
                ("mode", ctypes.c_uint32), ("device", ctypes.c_int),
                ("hbm_values_addr", ctypes.c_uint64), ("host_values_addr", ctypes.c_uint64)]


_lib = None


def _lib_or_none():
    return _lib


def load(path: str = LIB_PATH):
    """Load libhkv.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing; build it with "
                          "`python -m hash_table_cache_gb300._build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    u64, u32, vp, st = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_int
    sig = {
        "hkv_create": [u64, u32, u32, u64, ctypes.c_int, ctypes.POINTER(vp)],
        "hkv_destroy": [vp],
        "hkv_find": [vp, u64, vp, vp, vp, vp, vp],
        "hkv_insert_or_assign": [vp, u64, vp, vp, vp, vp],
        "hkv_insert_or_assign_noalloc": [vp, u64, vp, vp, vp, vp],
        "hkv_assign": [vp, u64, vp, vp, vp, vp],
        "hkv_insert_and_evict": [vp, u64, vp, vp, vp, vp, vp, vp, vp, vp],
        "hkv_find_or_insert": [vp, u64, vp, vp, vp, vp, vp],
        "hkv_contains": [vp, u64, vp, vp, vp],
        "hkv_find_ptr": [vp, u64, vp, vp, vp, vp, vp],
        "hkv_erase": [vp, u64, vp, vp],
        "hkv_size": [vp, ctypes.POINTER(u64), vp],
        "hkv_export": [vp, u64, u64, u64, vp, vp, vp, vp, vp],
        "hkv_get_error_counts": [vp, ctypes.POINTER(u64), ctypes.POINTER(u64)],
        "hkv_get_op_counts": [vp, ctypes.POINTER(OpCounts)],
        "hkv_reset_op_counts": [vp],
        "hkv_get_info": [vp, ctypes.POINTER(Info)],
        "hkv_set_epoch": [vp, u32],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = st
    lib.hkv_status_string.argtypes = [st]
    lib.hkv_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _p(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr() or None
    return int(x) or None


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream or None
    return int(stream) or None


# ---------------------------------------------------------------------------
# C ABI, one to one.
# ---------------------------------------------------------------------------
def hkv_create(capacity, dim, mode=HKV_MODE_SINGLE, value_hbm_bytes=0, device=0):
    """Returns (status, handle)."""
    h = ctypes.c_void_p()
    st = load().hkv_create(int(capacity), int(dim), int(mode), int(value_hbm_bytes), int(device),
                           ctypes.byref(h))
    return st, h.value


def hkv_destroy(table):
    return load().hkv_destroy(table)


def hkv_find(table, n, keys, values_out, found_out, scores_out=None, stream=None):
    return load().hkv_find(table, int(n), _p(keys), _p(values_out), _p(found_out), _p(scores_out),
                           _s(stream))


def hkv_insert_or_assign(table, n, keys, values, scores=None, stream=None):
    return load().hkv_insert_or_assign(table, int(n), _p(keys), _p(values), _p(scores), _s(stream))


def hkv_insert_or_assign_noalloc(table, n, keys, values, scores=None, stream=None):
    """insert_or_assign without any allocation by the library: its working
    memory is a fixed array inside libhkv.so (see include/hkv.h for the size
    limit, the sharing rule and the first-call set-up)."""
    return load().hkv_insert_or_assign_noalloc(table, int(n), _p(keys), _p(values), _p(scores),
                                               _s(stream))


def hkv_insert_and_evict(table, n, keys, values, scores, ev_keys, ev_values, ev_scores, ev_count,
                         stream=None):
    return load().hkv_insert_and_evict(table, int(n), _p(keys), _p(values), _p(scores), _p(ev_keys),
                                       _p(ev_values), _p(ev_scores), _p(ev_count), _s(stream))


def hkv_find_or_insert(table, n, keys, values_inout, scores, found_out, stream=None):
    return load().hkv_find_or_insert(table, int(n), _p(keys), _p(values_inout), _p(scores),
                                     _p(found_out), _s(stream))


def hkv_contains(table, n, keys, found_out, stream=None):
    return load().hkv_contains(table, int(n), _p(keys), _p(found_out), _s(stream))


def hkv_find_ptr(table, n, keys, ptrs_out, found_out, scores_out=None, stream=None):
    return load().hkv_find_ptr(table, int(n), _p(keys), _p(ptrs_out), _p(found_out),
                               _p(scores_out), _s(stream))


def hkv_assign(table, n, keys, values, scores=None, stream=None):
    return load().hkv_assign(table, int(n), _p(keys), _p(values), _p(scores), _s(stream))


def hkv_erase(table, n, keys, stream=None):
    return load().hkv_erase(table, int(n), _p(keys), _s(stream))


def hkv_size(table, stream=None):
    """Returns (status, size)."""
    v = ctypes.c_uint64()
    st = load().hkv_size(table, ctypes.byref(v), _s(stream))
    return st, int(v.value)


def hkv_export(table, slot_begin, slot_end, min_score, keys_out, values_out, scores_out, count_out,
               stream=None):
    return load().hkv_export(table, int(slot_begin), int(slot_end), int(min_score), _p(keys_out),
                             _p(values_out), _p(scores_out), _p(count_out), _s(stream))


def hkv_get_error_counts(table):
    """Returns (status, reserved_keys, timeouts)."""
    a, b = ctypes.c_uint64(), ctypes.c_uint64()
    st = load().hkv_get_error_counts(table, ctypes.byref(a), ctypes.byref(b))
    return st, int(a.value), int(b.value)


def hkv_get_op_counts(table):
    c = OpCounts()
    st = load().hkv_get_op_counts(table, ctypes.byref(c))
    return st, c.as_dict()


def hkv_reset_op_counts(table):
    return load().hkv_reset_op_counts(table)


def hkv_get_info(table):
    i = Info()
    st = load().hkv_get_info(table, ctypes.byref(i))
    return st, {f: getattr(i, f) for f, _ in Info._fields_}


def hkv_set_epoch(table, epoch):
    return load().hkv_set_epoch(table, int(epoch) & 0xFFFFFFFF)


def hkv_status_string(status):
    return load().hkv_status_string(int(status)).decode()


# ---------------------------------------------------------------------------
# Tensor-level convenience wrapper.
# ---------------------------------------------------------------------------
def _check(st, what):
    if st != HKV_OK:
        raise HKVError(st, what)


class HashTable:
    """One table on one device.  Keys and scores are int64 tensors holding the
    uint64 bits; values are float32 [n, dim]; all on the table's device."""

    def __init__(self, capacity, dim, mode=HKV_MODE_SINGLE, value_hbm_bytes=0, device=0):
        st, h = hkv_create(capacity, dim, mode, value_hbm_bytes, device)
        _check(st, "hkv_create")
        self.handle = h
        self.capacity = int(capacity)
        self.dim = int(dim)
        self.mode = int(mode)
        self.device = int(device)

    def close(self):
        if getattr(self, "handle", None):
            hkv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def num_buckets(self):
        return self.capacity // SLOTS_PER_BUCKET

    def find(self, keys, values_out=None, found_out=None, scores_out=None, with_scores=True,
             stream=None):
        import torch
        n = keys.numel()
        dev = keys.device
        if values_out is None:
            values_out = torch.zeros((n, self.dim), dtype=torch.float32, device=dev)
        if found_out is None:
            found_out = torch.empty(n, dtype=torch.uint8, device=dev)
        if scores_out is None and with_scores:
            scores_out = torch.zeros(n, dtype=torch.int64, device=dev)
        _check(hkv_find(self.handle, n, keys, values_out, found_out, scores_out, stream), "hkv_find")
        return values_out, found_out, scores_out

    def insert_or_assign(self, keys, values, scores=None, stream=None):
        _check(hkv_insert_or_assign(self.handle, keys.numel(), keys, values, scores, stream),
               "hkv_insert_or_assign")

    def insert_and_evict(self, keys, values, scores=None, stream=None):
        """Returns (evicted keys, values, scores) -- unsorted, on the device."""
        import torch
        n = keys.numel()
        dev = keys.device
        ek = torch.empty(max(n, 1), dtype=torch.int64, device=dev)
        ev = torch.empty((max(n, 1), self.dim), dtype=torch.float32, device=dev)
        es = torch.empty(max(n, 1), dtype=torch.int64, device=dev)
        cnt = torch.zeros(1, dtype=torch.int64, device=dev)
        _check(hkv_insert_and_evict(self.handle, n, keys, values, scores, ek, ev, es, cnt, stream),
               "hkv_insert_and_evict")
        c = int(cnt.item())
        return ek[:c], ev[:c], es[:c]

    def find_or_insert(self, keys, values_inout, scores=None, stream=None):
        """values_inout is updated in place; returns the found flags."""
        import torch
        found = torch.empty(keys.numel(), dtype=torch.uint8, device=keys.device)
        _check(hkv_find_or_insert(self.handle, keys.numel(), keys, values_inout, scores, found,
                                  stream), "hkv_find_or_insert")
        return found

    def contains(self, keys, stream=None):
        import torch
        found = torch.empty(keys.numel(), dtype=torch.uint8, device=keys.device)
        _check(hkv_contains(self.handle, keys.numel(), keys, found, stream), "hkv_contains")
        return found

    def find_ptr(self, keys, with_scores=True, stream=None):
        """Returns (row addresses as int64, found, scores)."""
        import torch
        n = keys.numel()
        ptrs = torch.empty(n, dtype=torch.int64, device=keys.device)
        found = torch.empty(n, dtype=torch.uint8, device=keys.device)
        scs = torch.empty(n, dtype=torch.int64, device=keys.device) if with_scores else None
        _check(hkv_find_ptr(self.handle, n, keys, ptrs, found, scs, stream), "hkv_find_ptr")
        return ptrs, found, scs

    def assign(self, keys, values, scores=None, stream=None):
        _check(hkv_assign(self.handle, keys.numel(), keys, values, scores, stream), "hkv_assign")

    def erase(self, keys, stream=None):
        _check(hkv_erase(self.handle, keys.numel(), keys, stream), "hkv_erase")

    def size(self, stream=None):
        st, v = hkv_size(self.handle, stream)
        _check(st, "hkv_size")
        return v

    def export(self, slot_begin=0, slot_end=None, min_score=0, with_values=True, stream=None):
        """Entries of slots [slot_begin, slot_end) with score >= min_score,
        sorted by key (as uint64).  Returns (keys, values, scores) tensors."""
        import torch
        slot_end = self.capacity if slot_end is None else min(int(slot_end), self.capacity)
        m = max(0, slot_end - slot_begin)
        dev = torch.device("cuda", self.device)
        keys = torch.empty(max(m, 1), dtype=torch.int64, device=dev)
        vals = torch.empty((max(m, 1), self.dim), dtype=torch.float32, device=dev) if with_values else None
        scs = torch.empty(max(m, 1), dtype=torch.int64, device=dev)
        cnt = torch.zeros(1, dtype=torch.int64, device=dev)
        _check(hkv_export(self.handle, slot_begin, slot_end, min_score, keys, vals, scs, cnt, stream),
               "hkv_export")
        c = int(cnt.item())
        keys, scs = keys[:c], scs[:c]
        vals = vals[:c] if vals is not None else None
        order = torch.argsort(keys.view(torch.int64) ^ (-(2 ** 63)))  # uint64 order
        return keys[order], (vals[order] if vals is not None else None), scs[order]

    def error_counts(self):
        st, r, t = hkv_get_error_counts(self.handle)
        if st not in (HKV_OK, HKV_ERR_RESERVED_KEY, HKV_ERR_TIMEOUT):
            _check(st, "hkv_get_error_counts")
        return {"reserved": r, "timeouts": t, "status": st}

    def op_counts(self):
        st, c = hkv_get_op_counts(self.handle)
        _check(st, "hkv_get_op_counts")
        return c

    def reset_op_counts(self):
        _check(hkv_reset_op_counts(self.handle), "hkv_reset_op_counts")

    def info(self):
        st, i = hkv_get_info(self.handle)
        _check(st, "hkv_get_info")
        return i

    def set_epoch(self, epoch):
        _check(hkv_set_epoch(self.handle, epoch), "hkv_set_epoch")
