"""CPU checks of the benchmark's byte models and bookkeeping: the algorithmic
bytes per find key against the per-path figures of the HKV find (Algorithm 1:
key, digest line, expected key confirms, value row in and out, flag, score),
the insert_or_assign byte count, the random-access floors in limiting cases,
and the rule that a stored ncu traffic figure is reported only while the
kernel sources it was taken from are unchanged."""
import hashlib
import math
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_find_bytes_per_key_paths():
    # miss: key 8 + digest line 128 + half a key confirm (128/256 * 8) + flag 1
    assert bench.find_bytes_per_key(32, 0.0) == pytest.approx(8 + 128 + 4 + 1)
    # hit: key, line, 1 + 127/256 confirms, row read and row write, flag,
    # score read and write
    for dim in (8, 32, 64, 128):
        hit = 8 + 128 + 8 * (1 + 127 / 256) + 2 * 4 * dim + 1 + 16
        assert bench.find_bytes_per_key(dim, 1.0) == pytest.approx(hit)
    # the 80%-hit mix at dim 32 is the weighted sum, about 365 bytes
    mix = bench.find_bytes_per_key(32, 0.8)
    assert mix == pytest.approx(0.8 * bench.find_bytes_per_key(32, 1.0)
                                + 0.2 * bench.find_bytes_per_key(32, 0.0))
    assert 364 < mix < 366


def test_upsert_bytes_terms():
    # one key, one touched bucket, one written row, dim 4 (16-byte rows)
    assert bench.upsert_bytes(1, 4, 1, 1, False) == (8 + 16) + (2048 + 256) + (16 + 16)
    assert bench.upsert_bytes(1, 4, 1, 1, True) == bench.upsert_bytes(1, 4, 1, 1, False) + 8
    # linear in each count
    a = bench.upsert_bytes(10, 32, 3, 7, False)
    b = bench.upsert_bytes(20, 32, 6, 14, False)
    assert b == 2 * a
    assert bench.upsert_bytes(0, 32, 0, 0, True) == 0


def test_find_access_floor_limits():
    rates = {32: 1e9, 128: 1e9}
    huge_bw = 1e30  # streamed bytes cost nothing
    n, nb = 1 << 16, 1 << 10
    # all misses: half a sector per key plus one line per touched bucket
    t0 = bench.find_access_floor(n, 32, 0.0, nb, rates, huge_bw)
    lines = nb * (1 - math.exp(-n / nb))
    assert t0 == pytest.approx(n * 0.5 / 1e9 + lines / 1e9)
    # all hits at dim 32 (128-byte rows): 1 + 127/256 sectors and a row per key
    t1 = bench.find_access_floor(n, 32, 1.0, nb, rates, huge_bw)
    assert t1 == pytest.approx(n * (1 + 127 / 256) / 1e9 + n / 1e9 + lines / 1e9)
    # streamed bytes add at the copy bandwidth
    t2 = bench.find_access_floor(n, 32, 1.0, nb, rates, 1.0)  # 1 GB/s
    assert t2 - t1 == pytest.approx(n * (8 + 4 * 32 + 8 + 1) / 1e9, rel=1e-6)


def test_upsert_access_floor_monotone():
    rates = {32: 4e10, 128: 2e10}
    base = bench.upsert_access_floor(1 << 20, 32, 1 << 19, 1 << 15, rates, 6000.0)
    assert base > 0
    assert bench.upsert_access_floor(1 << 20, 32, 1 << 20, 1 << 15, rates, 6000.0) > base
    assert bench.upsert_access_floor(1 << 20, 32, 1 << 19, 1 << 16, rates, 6000.0) > base


def test_ncu_traffic_follows_sources(monkeypatch):
    files = ("find.cu", "common.cuh", "launch.h")
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "hash_table_cache_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    good = {"bytes": 1234, "sources": files, "sha256": h.hexdigest()[:16]}
    monkeypatch.setitem(bench.NCU_TRAFFIC, "probe_kernel", good)
    assert bench.ncu_traffic("probe_kernel") == 1234
    stale = dict(good, sha256="0" * 16)
    monkeypatch.setitem(bench.NCU_TRAFFIC, "probe_kernel", stale)
    assert bench.ncu_traffic("probe_kernel") is None
    assert bench.ncu_traffic("no_such_kernel") is None
