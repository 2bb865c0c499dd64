"""GPU parity of the cache-workflow operations: insert_and_evict and
find_or_insert (HKV §4.1), contains (HKV §3.5) and the pointer-returning
find* (HKV §5.2-§5.3), against the oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.gpu_util import assert_same_state, dkeys, dvals, read_device, table_state, u64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hkv():
    import hash_table_cache_gb300 as m
    from hash_table_cache_gb300 import _build
    _build.build()
    m.load()
    return m


@pytest.fixture(scope="module")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.mark.parametrize("num_buckets,dim,tiered", [(1, 4, False), (16, 8, False), (300, 3, False),
                                                    (16, 8, True), (300, 4, True)])
def test_insert_and_evict_and_find_or_insert(hkv, oracle_mod, num_buckets, dim, tiered):
    """tiered: the rows of buckets past the first half live in host memory,
    so evicted rows are copied out of it (still equal to the oracle)."""
    rng = np.random.default_rng(num_buckets)
    cap = num_buckets * 128
    t = (hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_TIERED,
                       value_hbm_bytes=(num_buckets // 2) * 128 * 4 * dim)
         if tiered else hkv.HashTable(cap, dim))
    o = oracle_mod.OracleTable(num_buckets, dim)
    universe = wl.unique_keys(500 + num_buckets, 3 * cap)
    for step in range(16):
        n = int(rng.integers(1, 2 * cap))
        keys = universe[rng.integers(0, universe.size, n)]
        vals = rng.standard_normal((n, dim)).astype(np.float32)
        scores = rng.integers(0, 60, n).astype(np.uint64) if step % 3 else None
        ds = None if scores is None else dkeys(scores)
        if step % 2 == 0:
            ek, ev, es = t.insert_and_evict(dkeys(keys), dvals(vals), ds)
            torch.cuda.synchronize()
            c, (ok_, ov, os_) = o.insert_and_evict(keys, vals, scores)
            ek = u64(ek)
            order = np.argsort(ek)
            assert np.array_equal(ek[order], ok_)
            assert np.array_equal(u64(es)[order], os_)
            assert np.array_equal(ev.cpu().numpy()[order].view(np.uint32), ov.view(np.uint32))
        else:
            gv = dvals(vals)
            gf = t.find_or_insert(dkeys(keys), gv, ds)
            torch.cuda.synchronize()
            c, ov, of = o.find_or_insert(keys, vals, scores)
            assert np.array_equal(gf.cpu().numpy(), of)
            assert np.array_equal(gv.cpu().numpy().view(np.uint32), ov.view(np.uint32))
        assert_same_state(t, o)
        assert t.size() == o.size()
    t.close()


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_contains_and_find_ptr(hkv, oracle_mod, mode):
    B, dim = 64, 8
    cap = B * 128
    kw = {"value_hbm_bytes": (B // 2) * 128 * 4 * dim} if mode == 2 else {}
    t = hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_TIERED if mode == 2 else mode, **kw)
    o = oracle_mod.OracleTable(B, dim, dual=mode == 1)
    keys = wl.unique_keys(600, cap)
    vals = wl.key_values(keys, dim, salt=3)
    sc = np.arange(keys.size, dtype=np.uint64)
    t.insert_or_assign(dkeys(keys), dvals(vals), dkeys(sc))
    o.insert_or_assign(keys, vals, sc)
    q = np.concatenate([keys[::2], wl.unique_keys(601, 3000)])
    if mode == 1:
        # dual placement depends on processing order: compare with the GPU
        # table's own contents (its find is checked against them elsewhere)
        gv_, gf_, gs_ = t.find(dkeys(q))
        torch.cuda.synchronize()
        ov, of, os_ = gv_.cpu().numpy(), gf_.cpu().numpy(), u64(gs_)
        rk = set(u64(t.export(with_values=False)[0]).tolist())
        assert np.array_equal(of.astype(bool), np.array([int(x) in rk for x in q]))
        # independent of the GPU: keys never inserted are not found, a found
        # key carries the value and score it was inserted with, and every
        # resident key (all of them inserted keys, every other one queried)
        # is found
        n_ins = keys[::2].size
        assert not of[n_ins:].any()
        pos = {int(k): j for j, k in enumerate(keys)}
        src = np.array([pos[int(x)] for x in q[:n_ins]])
        fi = np.flatnonzero(of[:n_ins])
        assert np.array_equal(ov[fi].view(np.uint32), vals[src[fi]].view(np.uint32))
        assert np.array_equal(os_[fi], sc[src[fi]])
        assert len(rk) == t.size() and rk <= set(int(k) for k in keys)
        assert of[:n_ins].sum() == len(rk & set(int(k) for k in keys[::2]))
    else:
        ov, of, os_ = o.find(q)
    gf = t.contains(dkeys(q))
    torch.cuda.synchronize()
    assert np.array_equal(gf.cpu().numpy(), of)
    ptrs, pf, ps = t.find_ptr(dkeys(q))
    torch.cuda.synchronize()
    pf = pf.cpu().numpy()
    assert np.array_equal(pf, of)
    hit = of.astype(bool)
    assert np.array_equal(u64(ps)[hit], os_[hit])
    p = ptrs.cpu().numpy()
    assert np.all(p[~hit] == 0) and np.all(p[hit] % 16 == 0)
    assert np.unique(p[hit]).size == hit.sum()
    for i in np.flatnonzero(hit)[:400]:
        row = read_device(p[i], 4 * dim).view(np.float32)
        assert np.array_equal(row, ov[i])
    t.close()


@pytest.mark.parametrize("tiered", [False, True])
def test_export_score_threshold(hkv, oracle_mod, tiered):
    """export with a score threshold (HKV §4.1 export_batch_if, predicate
    score >= threshold; DynamicEmb incremental_dump): for thresholds from 0
    past the largest score, over the whole table and over bucket ranges, the
    entries equal the oracle's bit for bit (keys, values, scores)."""
    B, dim = 96, 6
    cap = B * 128
    kw = {"mode": hkv.HKV_MODE_TIERED, "value_hbm_bytes": (B // 3) * 128 * 4 * dim} if tiered else {}
    t = hkv.HashTable(cap, dim, **kw)
    o = oracle_mod.OracleTable(B, dim)
    rng = np.random.default_rng(9)
    keys = wl.unique_keys(710, int(1.3 * cap))
    for lo in range(0, keys.size, 3000):
        k = keys[lo:lo + 3000]
        v = wl.key_values(k, dim, salt=lo)
        sc = rng.integers(0, 1000, k.size).astype(np.uint64)
        t.insert_or_assign(dkeys(k), dvals(v), dkeys(sc))
        o.insert_or_assign(k, v, sc)
    torch.cuda.synchronize()
    for thr in (0, 1, 500, 990, 999, 1000, 1 << 62):
        for b0, b1 in ((0, B), (0, 1), (17, 18), (40, 71), (B - 1, B)):
            gk, gv, gs = table_state(t, b0 * 128, b1 * 128, thr)
            ok, ov, os_ = o.export(b0, b1, thr)
            assert np.array_equal(gk, ok), (thr, b0, b1)
            assert np.array_equal(gs, os_)
            assert np.array_equal(gv.view(np.uint32), ov.view(np.uint32))
            assert np.all(gs >= thr)
    t.close()
