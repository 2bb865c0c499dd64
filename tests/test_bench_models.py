"""CPU checks of the benchmark's byte models and bookkeeping: the algorithmic
bytes per find key against the per-path figures of the HKV find (Algorithm 1:
key, digest line, expected key confirms, value row in and out, flag, score),
the insert_or_assign byte counts (slot layout and per-path), the dual-mode
find bytes, the random-access floors in limiting cases, the hash the bench
uses to split dual-mode hits (equal to the oracle's buckets), the mapping of
find* addresses to rows,
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
    rates = {32: {"plateau": 1e9}, 128: {"plateau": 1e9}}
    huge_bw = 1e30  # streamed bytes cost nothing
    n, nb = 1 << 16, 1 << 10
    lines = nb * (1 - math.exp(-n / nb))
    # all misses: half a sector per key plus one line per touched bucket
    c0 = bench.find_random_counts(n, 32, 0.0, nb)
    assert bench.access_floor(c0, 0, rates, huge_bw) == pytest.approx(n * 0.5 / 1e9 + lines / 1e9)
    # all hits at dim 32 (128-byte rows): 1 + 127/256 sectors and a row per key
    c1 = bench.find_random_counts(n, 32, 1.0, nb)
    t1 = bench.access_floor(c1, 0, rates, huge_bw)
    assert t1 == pytest.approx(n * (1 + 127 / 256) / 1e9 + n / 1e9 + lines / 1e9)
    # streamed bytes add at the copy bandwidth
    t2 = bench.access_floor(c1, 1e9, rates, 1.0)  # 1 GB at 1 GB/s
    assert t2 - t1 == pytest.approx(1.0)
    # rows wider than 128 bytes are counted at their own granule's rate
    c3 = bench.find_random_counts(n, 64, 1.0, nb)
    assert c3[256] == n and c3[32] == pytest.approx(n * (1 + 127 / 256))


def test_upsert_bytes_paths():
    d = 4 * 32
    one = dict(updated=0, admitted=0, evicted=0, rejected=0)
    # each path alone, one key
    assert bench.upsert_bytes_paths(dict(one, updated=1), 1, 32) == 164 + 2 * d
    assert bench.upsert_bytes_paths(dict(one, admitted=1), 1, 32) == 165 + 2 * d
    assert bench.upsert_bytes_paths(dict(one, admitted=1, evicted=1), 1, 32) == 1189 + 2 * d
    assert bench.upsert_bytes_paths(dict(one, rejected=1), 1, 32) == 1172
    # a repeated key of the batch costs its key and row only
    assert bench.upsert_bytes_paths(dict(one, updated=1), 2, 32) == 164 + 2 * d + 8 + d
    # dual mode: the second bucket's line, and a second score scan on D2
    assert bench.upsert_bytes_paths(dict(one, admitted=1), 1, 32, dual=True) == 165 + 2 * d + 132
    assert bench.upsert_bytes_paths(dict(one, admitted=1, evicted=1), 1, 32,
                                    dual=True) == 2345 + 2 * d
    assert bench.upsert_bytes_paths(dict(one, rejected=1), 1, 32, dual=True) == 1172 + 1156


def test_find_bytes_dual():
    hit = bench.find_bytes_per_key(128, 1.0)
    miss = bench.find_bytes_per_key(128, 0.0)
    assert bench.find_bytes_dual(128, 1, 0, 0) == pytest.approx(hit)
    assert bench.find_bytes_dual(128, 0, 1, 0) == pytest.approx(hit + 132)
    assert bench.find_bytes_dual(128, 0, 0, 1) == pytest.approx(miss + 132)


def test_measurement_hash_is_the_documented_hash(oracle_mod):
    """The bench splits dual-mode hits by bucket with the hash the header
    documents; it must give the oracle's buckets (both candidates, the b1 =
    b2 rule included)."""
    import numpy as np
    import torch
    import workloads as wl
    nb = 1 << 10
    o = oracle_mod.OracleTable(nb, 4, dual=True)
    k = wl.unique_keys(5, 200000)
    kt = torch.from_numpy(wl.as_i64(k))
    b1 = bench.first_bucket_t(kt, nb).numpy().astype(np.uint64)
    b2 = bench.second_bucket_t(kt, bench.first_bucket_t(kt, nb), nb).numpy().astype(np.uint64)
    assert np.array_equal(b1, o.buckets_of(k, 0))
    assert np.array_equal(b2, o.buckets_of(k, 1))
    assert (b1 == b2).sum() == 0


def test_rows_of_ptrs():
    import torch
    info = {"dim": 4, "hbm_value_rows": 256, "hbm_values_addr": 1 << 20,
            "host_values_addr": 1 << 40}
    rows = torch.tensor([0, 5, 255, 256, 300, 7])
    found = torch.tensor([1, 1, 1, 1, 1, 0], dtype=torch.uint8)
    ptrs = torch.where(rows < 256, (1 << 20) + rows * 16, (1 << 40) + (rows - 256) * 16)
    got = bench.rows_of_ptrs(ptrs, found, info)
    assert got[:5].tolist() == [0, 5, 255, 256, 300]
    assert got[5].item() == 0  # not found


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


def test_slab_threshold_matches_the_header():
    """The bench probes a tiered slab's memory the way the library allocates
    it: the size threshold is the header's HKV_HOST_SLAB_MAPPED_MAX."""
    import re
    text = open(os.path.join(ROOT, "include", "hkv.h")).read()
    m = re.search(r"#define HKV_HOST_SLAB_MAPPED_MAX \((\d+)ull << (\d+)\)", text)
    assert m and bench.HOST_SLAB_MAPPED_MAX == int(m.group(1)) << int(m.group(2))
    assert bench.slab_kinds(bench.HOST_SLAB_MAPPED_MAX) == (2, 3)
    assert bench.slab_kinds(bench.HOST_SLAB_MAPPED_MAX + 1) == (6, 7)
