"""Python handle on the CPU oracle (``hkv_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` are the only callers.  The library in
``hash_table_cache_gb300/`` never imports this package.

The oracle follows "HierarchicalKV: A GPU Hash Table with Cache Semantics for
Continuous Online Embedding Storage" (arXiv 2603.17168v1): Algorithm 1 (find),
Algorithm 2 (single-bucket upsert with admission and eviction), Algorithm 3
(score-based dual-bucket upsert), and the reader/updater/inserter operations of
§3.5.  The readings it takes where the paper is silent are listed at the top
of ``hkv_oracle.cpp``.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against brute force, closed forms and the paper's special cases, except the
hash (``hash64``), which the paper names only as a Murmur3 derivative; it is
pinned by bijectivity and avalanche statistics only.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hkv_oracle.cpp")
_LIB = os.path.join(_HERE, "libhkv_oracle.so")

RESERVED_LO = 0xFFFFFFFFFFFFFFF0
SLOTS = 128

# Score policies (reading R10 in hkv_oracle.cpp; HKV §3.3, Table 8 names).
POLICY_CUSTOMIZED, POLICY_LRU, POLICY_LFU, POLICY_EPOCH_LRU, POLICY_EPOCH_LFU = range(5)


class _Counts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("updated", "admitted", "evicted", "rejected", "reserved", "filtered", "erased")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler (plain -O2, no CUDA)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", _SRC, "-o", tmp],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    u64, u32, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p
    sig = {
        "oracle_create": (vp, [u64, u32, ctypes.c_int, u32]),
        "oracle_set_epoch": (None, [vp, u32]),
        "oracle_destroy": (None, [vp]),
        "oracle_set_bucket_filter": (ctypes.c_int, [vp, u64, vp]),
        "oracle_hash": (u64, [u64]),
        "oracle_bucket": (u64, [vp, u64, ctypes.c_int]),
        "oracle_step": (u64, [vp]),
        "oracle_buckets": (None, [vp, u64, vp, ctypes.c_int, vp]),
        "oracle_insert_or_assign": (None, [vp, u64, vp, vp, vp, ctypes.POINTER(_Counts)]),
        "oracle_assign": (None, [vp, u64, vp, vp, vp, ctypes.POINTER(_Counts)]),
        "oracle_erase": (None, [vp, u64, vp, ctypes.POINTER(_Counts)]),
        "oracle_find": (u64, [vp, u64, vp, vp, vp, vp]),
        "oracle_insert_and_evict": (None, [vp, u64, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(_Counts)]),
        "oracle_find_or_insert": (None, [vp, u64, vp, vp, vp, vp, ctypes.POINTER(_Counts)]),
        "oracle_contains": (None, [vp, u64, vp, vp]),
        "oracle_size": (u64, [vp]),
        "oracle_bucket_size": (u64, [vp, u64]),
        "oracle_export": (u64, [vp, u64, u64, u64, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _keys(a):
    return np.ascontiguousarray(a, dtype=np.uint64)


def hash64(key: int) -> int:
    """H(k): the 64-bit MurmurHash3 finalizer (reading R1)."""
    return int(_load().oracle_hash(ctypes.c_uint64(int(key))))


class OracleTable:
    """Single-threaded model of one table (single or dual-bucket mode) under
    one score policy (POLICY_*)."""

    def __init__(self, num_buckets: int, dim: int, dual: bool = False,
                 policy: int = POLICY_CUSTOMIZED):
        lib = _load()
        self.num_buckets = int(num_buckets)
        self.dim = int(dim)
        self.dual = bool(dual)
        self.policy = int(policy)
        self._h = lib.oracle_create(self.num_buckets, self.dim, int(self.dual), self.policy)
        if not self._h:
            raise ValueError("oracle_create rejected the arguments")

    def set_epoch(self, epoch: int):
        _load().oracle_set_epoch(self._h, int(epoch) & 0xFFFFFFFF)

    def _scores(self, scores):
        if scores is None:
            return None
        if self.policy in (POLICY_LRU, POLICY_EPOCH_LRU):
            raise ValueError("clock-driven policies take no caller scores")
        return _keys(scores)

    def close(self):
        if self._h:
            _load().oracle_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def capacity(self):
        return self.num_buckets * SLOTS

    @property
    def step(self):
        return int(_load().oracle_step(self._h))

    def set_bucket_filter(self, buckets):
        b = _keys(buckets)
        if _load().oracle_set_bucket_filter(self._h, b.size, _ptr(b)) != 0:
            raise ValueError("bucket filter needs single-bucket mode")

    def bucket(self, key: int, which: int = 0) -> int:
        return int(_load().oracle_bucket(self._h, int(key), int(which)))

    def buckets_of(self, keys, which: int = 0) -> np.ndarray:
        k = _keys(keys)
        out = np.zeros(k.size, np.uint64)
        _load().oracle_buckets(self._h, k.size, _ptr(k), int(which), _ptr(out))
        return out

    def _values(self, values, n):
        v = np.ascontiguousarray(values, dtype=np.float32)
        if v.size != n * self.dim:
            raise ValueError("values must hold n * dim float32")
        return v

    def insert_or_assign(self, keys, values, scores=None) -> dict:
        k = _keys(keys)
        v = self._values(values, k.size)
        s = self._scores(scores)
        c = _Counts()
        _load().oracle_insert_or_assign(self._h, k.size, _ptr(k), _ptr(v), _ptr(s), ctypes.byref(c))
        return c.as_dict()

    def assign(self, keys, values, scores=None) -> dict:
        k = _keys(keys)
        v = self._values(values, k.size)
        s = self._scores(scores)
        c = _Counts()
        _load().oracle_assign(self._h, k.size, _ptr(k), _ptr(v), _ptr(s), ctypes.byref(c))
        return c.as_dict()

    def erase(self, keys) -> dict:
        k = _keys(keys)
        c = _Counts()
        _load().oracle_erase(self._h, k.size, _ptr(k), ctypes.byref(c))
        return c.as_dict()

    def find(self, keys, values_out=None, scores_out=None):
        """Returns (values, found, scores); untouched rows keep values_out/scores_out."""
        k = _keys(keys)
        n = k.size
        vals = np.zeros((n, self.dim), np.float32) if values_out is None else values_out
        scs = np.zeros(n, np.uint64) if scores_out is None else scores_out
        found = np.zeros(n, np.uint8)
        _load().oracle_find(self._h, n, _ptr(k), _ptr(vals), _ptr(found), _ptr(scs))
        return vals, found, scs

    def insert_and_evict(self, keys, values, scores=None):
        """Returns (counts, (evicted keys, values, scores) sorted by key)."""
        k = _keys(keys)
        v = self._values(values, k.size)
        s = self._scores(scores)
        ek = np.zeros(max(k.size, 1), np.uint64)
        ev = np.zeros((max(k.size, 1), self.dim), np.float32)
        es = np.zeros(max(k.size, 1), np.uint64)
        cnt = np.zeros(1, np.uint64)
        c = _Counts()
        _load().oracle_insert_and_evict(self._h, k.size, _ptr(k), _ptr(v), _ptr(s), _ptr(ek), _ptr(ev),
                                        _ptr(es), _ptr(cnt), ctypes.byref(c))
        m = int(cnt[0])
        return c.as_dict(), (ek[:m], ev[:m], es[:m])

    def find_or_insert(self, keys, values, scores=None):
        """Returns (counts, values after the call, found flags)."""
        k = _keys(keys)
        v = self._values(values, k.size).copy().reshape(k.size, self.dim)
        s = self._scores(scores)
        found = np.zeros(k.size, np.uint8)
        c = _Counts()
        _load().oracle_find_or_insert(self._h, k.size, _ptr(k), _ptr(v), _ptr(s), _ptr(found),
                                      ctypes.byref(c))
        return c.as_dict(), v, found

    def contains(self, keys):
        k = _keys(keys)
        found = np.zeros(k.size, np.uint8)
        _load().oracle_contains(self._h, k.size, _ptr(k), _ptr(found))
        return found

    def size(self) -> int:
        return int(_load().oracle_size(self._h))

    def bucket_size(self, b: int) -> int:
        return int(_load().oracle_bucket_size(self._h, int(b)))

    def export(self, b_begin=0, b_end=None, min_score=0):
        """Entries of buckets [b_begin, b_end) with score >= min_score, sorted by key."""
        lib = _load()
        b_end = self.num_buckets if b_end is None else b_end
        n = int(lib.oracle_export(self._h, b_begin, b_end, min_score, None, None, None))
        keys = np.zeros(n, np.uint64)
        vals = np.zeros((n, self.dim), np.float32)
        scs = np.zeros(n, np.uint64)
        lib.oracle_export(self._h, b_begin, b_end, min_score, _ptr(keys), _ptr(vals), _ptr(scs))
        return keys, vals, scs
