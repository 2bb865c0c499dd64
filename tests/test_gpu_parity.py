"""GPU parity: the CUDA library against the CPU oracle on the same seeded
inputs, through the C ABI.  Single-bucket results are compared bit-exactly."""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.gpu_util import DEV, assert_same_state, dkeys, dvals, find_compare, table_state

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


def test_c1_insert_then_find(hkv, oracle_mod):
    """Capacity 65,536 (512 buckets), dim 8, values N(0,1) seed 0: one batch of
    65,536 unique keys scored by insertion index, then one find batch of the
    even-indexed inserted keys plus as many fresh keys."""
    cap, dim, n = 65536, 8, 65536
    keys = wl.unique_keys(1, n)
    scores = np.arange(n, dtype=np.uint64)
    vals = wl.randn_values(0, n, dim).numpy()
    t = hkv.HashTable(cap, dim)
    o = oracle_mod.OracleTable(cap // 128, dim)
    t.insert_or_assign(dkeys(keys), dvals(vals), dkeys(scores))
    oc = o.insert_or_assign(keys, vals, scores)
    assert_same_state(t, o)
    gc = t.op_counts()
    for f in ("updated", "admitted", "evicted", "rejected"):
        assert gc[f] == oc[f], (f, gc, oc)
    assert t.size() == o.size()
    q = np.empty(n, np.uint64)
    q[0::2] = keys[0::2]
    q[1::2] = wl.unique_keys(2, n // 2)
    hits = find_compare(t, o, q)
    assert 0 < hits <= n // 2


@pytest.mark.parametrize("num_buckets,dim", [(1, 1), (1, 8), (3, 5), (64, 4), (100, 8), (37, 33),
                                             (5, 256), (3, 1001)])
@pytest.mark.parametrize("seed", [0, 1])
def test_random_ops_bit_exact(hkv, oracle_mod, num_buckets, dim, seed):
    """Random mixes of insert_or_assign (per-key scores with many ties, or the
    step counter), assign, erase and find, with duplicate and reserved keys;
    full table state compared after every call."""
    rng = np.random.default_rng(seed)
    cap = num_buckets * 128
    t = hkv.HashTable(cap, dim)
    o = oracle_mod.OracleTable(num_buckets, dim)
    universe = wl.unique_keys(seed + 77, 3 * cap)
    for step in range(25):
        op = rng.choice(["ioa", "ioa", "ioa", "ioa_step", "assign", "erase", "find"])
        n = int(rng.integers(0, 2 * cap + 2))
        keys = universe[rng.integers(0, universe.size, n)]
        if n and rng.random() < 0.3:
            keys[rng.integers(0, n)] = hkv.RESERVED_KEY_LO + int(rng.integers(0, 16))
        vals = rng.standard_normal((n, dim)).astype(np.float32)
        scores = rng.integers(0, 50, n).astype(np.uint64)
        if op in ("ioa", "ioa_step"):
            s = scores if op == "ioa" else None
            t.reset_op_counts()
            t.insert_or_assign(dkeys(keys), dvals(vals), None if s is None else dkeys(s))
            oc = o.insert_or_assign(keys, vals, s)
            gc = t.op_counts()
            for f in ("updated", "admitted", "evicted", "rejected"):
                assert gc[f] == oc[f], (step, f, gc, oc)
        elif op == "assign":
            s = scores if rng.random() < 0.5 else None
            t.assign(dkeys(keys), dvals(vals), None if s is None else dkeys(s))
            o.assign(keys, vals, s)
        elif op == "erase":
            t.erase(dkeys(keys))
            o.erase(keys)
        else:
            find_compare(t, o, keys)
        assert_same_state(t, o)
        assert t.size() == o.size()
    errs = t.error_counts()
    assert errs["timeouts"] == 0


@pytest.mark.parametrize("policy", ["custom", "lfu"])
@pytest.mark.parametrize("num_buckets,dim", [(64, 8), (300, 4), (1024, 16), (64, 260)])
def test_sparse_batches_bit_exact(hkv, oracle_mod, policy, num_buckets, dim):
    """Batches of at most four keys per bucket (the sparse path: one tile per
    touched bucket, the general kernel for the buckets it defers), on tables
    from empty to full: free-slot placement, one or two evictions per full
    bucket, resident keys beside absent ones, ties of score (small score
    range, or the step counter), repeated keys (last occurrence wins) and
    reserved keys; the whole table, the counts and a find compared with the
    oracle after every call."""
    rng = np.random.default_rng(num_buckets + dim)
    cap = num_buckets * 128
    mode = hkv.HKV_POLICY_LFU if policy == "lfu" else 0
    t = hkv.HashTable(cap, dim, mode=mode)
    o = oracle_mod.OracleTable(num_buckets, dim,
                               policy=oracle_mod.POLICY_LFU if policy == "lfu" else 0)
    universe = wl.unique_keys(num_buckets + 991, 3 * cap)
    for step in range(40):
        n = int(rng.integers(1, 4 * num_buckets + 1))
        if step < 8:  # fill with fresh keys first, then mixes
            keys = universe[step * (cap // 4):step * (cap // 4) + n]
        else:
            keys = universe[rng.integers(0, universe.size, n)]
        if rng.random() < 0.3:
            keys[rng.integers(0, n)] = hkv.RESERVED_KEY_LO + int(rng.integers(0, 16))
        if rng.random() < 0.3:
            keys[rng.integers(0, n, max(1, n // 8))] = keys[0]  # repeats
        vals = rng.standard_normal((n, dim)).astype(np.float32)
        r = rng.random()
        scores = None if r < 0.3 else rng.integers(0, 4 if r < 0.6 else 1 << 40, n).astype(np.uint64)
        t.reset_op_counts()
        t.insert_or_assign(dkeys(keys), dvals(vals), None if scores is None else dkeys(scores))
        oc = o.insert_or_assign(keys, vals, scores)
        gc = t.op_counts()
        for f in ("updated", "admitted", "evicted", "rejected"):
            assert gc[f] == oc[f], (step, f, gc, oc)
        assert_same_state(t, o)
        assert t.size() == o.size()
        if step % 5 == 4:
            q = np.concatenate([universe[rng.integers(0, universe.size, 500)],
                                wl.unique_keys(num_buckets + 5, 100, step * 100)])
            find_compare(t, o, q)
    t.close()


def test_c2_lambda_sweep(hkv, oracle_mod):
    """Capacity 2^22, dim 32: fill with unique keys in batches of 2^16 scored by
    the step counter; at load factor 0.50, 0.75, 0.90 and 1.00 compare a find
    batch of 2^20 keys (80% drawn from the residents, 20% fresh) bit-exactly;
    compare the whole table at 1.00, then an upsert batch of the same mix."""
    cap, dim, bs = 1 << 22, 32, 1 << 16
    t = hkv.HashTable(cap, dim)
    o = oracle_mod.OracleTable(cap // 128, dim)
    keys = wl.unique_keys(3, 2 * cap)
    pos = 0
    for lam in (0.5, 0.75, 0.9, 1.0):
        while o.size() < lam * cap and pos < keys.size:
            k = keys[pos:pos + bs]
            v = wl.key_values(k, dim, salt=1)
            t.insert_or_assign(dkeys(k), dvals(v), None)
            o.insert_or_assign(k, v, None)
            pos += bs
        assert t.size() == o.size()
        res = o.export()[0]
        q, _ = wl.hit_mix(4, res, 5, 1 << 20, 0.8, fresh_start=int(lam * 1000) << 20)
        hits = find_compare(t, o, q)
        assert hits >= 0.79 * q.size
    assert_same_state(t, o)
    res = o.export()[0]
    q, _ = wl.hit_mix(6, res, 7, 1 << 20, 0.8)
    v = wl.key_values(q, dim, salt=2)
    t.reset_op_counts()
    t.insert_or_assign(dkeys(q), dvals(v), None)
    oc = o.insert_or_assign(q, v, None)
    gc = t.op_counts()
    for f in ("updated", "admitted", "evicted", "rejected"):
        assert gc[f] == oc[f], (f, gc, oc)
    assert_same_state(t, o)


def test_edge_cases(hkv, oracle_mod):
    t = hkv.HashTable(256, 4)
    o = oracle_mod.OracleTable(2, 4)
    e = torch.empty(0, dtype=torch.int64, device=DEV)
    t.insert_or_assign(e, torch.empty((0, 4), device=DEV), e)
    t.find(e)
    t.erase(e)
    assert t.size() == 0
    # one key repeated: the last occurrence wins
    k = np.full(5000, 12345, np.uint64)
    v = np.arange(20000, dtype=np.float32).reshape(5000, 4)
    s = np.arange(5000, dtype=np.uint64)[::-1].copy()
    t.insert_or_assign(dkeys(k), dvals(v), dkeys(s))
    o.insert_or_assign(k, v, s)
    assert_same_state(t, o)
    # reserved keys only
    r = np.array([hkv.RESERVED_KEY_LO, 2**64 - 1, 2**64 - 2], np.uint64)
    t.insert_or_assign(dkeys(r), dvals(np.ones((3, 4))), None)
    find_compare(t, o, r)
    assert t.error_counts()["reserved"] >= 6
    assert_same_state(t, o)


@pytest.mark.parametrize("mode", ["single", "dual", "tiered"])
def test_empty_and_oversized_batches(hkv, mode):
    """n = 0 is a valid batch for every batched call in every mode and changes
    nothing; n above HKV_MAX_BATCH is refused with HKV_ERR_INVALID before any
    pointer is used; dual mode refuses insert_and_evict and find_or_insert
    whatever n is (HKV §7: its calls are find and insert_or_assign)."""
    B, dim = 64, 4
    cap = B * 128
    m = {"single": 0, "dual": hkv.HKV_MODE_DUAL, "tiered": hkv.HKV_MODE_TIERED}[mode]
    kw = {"value_hbm_bytes": (B // 2) * 128 * 4 * dim} if mode == "tiered" else {}
    t = hkv.HashTable(cap, dim, mode=m, **kw)
    k = dkeys(wl.unique_keys(700, 3000))
    t.insert_or_assign(k, wl.key_values_torch(k, dim, salt=1), None)
    torch.cuda.synchronize()
    before = table_state(t)
    s0, c0 = t.size(), t.op_counts()
    h, OK, INV = t.handle, hkv.HKV_OK, hkv.HKV_ERR_INVALID
    ev_keys = torch.zeros(1, dtype=torch.int64, device=DEV)
    ev_count = torch.zeros(1, dtype=torch.int64, device=DEV)
    dual = mode == "dual"
    for n, want in ((0, OK), (hkv.HKV_MAX_BATCH + 1, INV)):
        assert hkv.hkv_find(h, n, None, None, None) == want
        assert hkv.hkv_contains(h, n, None, None) == want
        assert hkv.hkv_find_ptr(h, n, None, None, None) == want
        assert hkv.hkv_insert_or_assign(h, n, None, None) == want
        assert hkv.hkv_insert_or_assign_noalloc(h, n, None, None) == want
        assert hkv.hkv_assign(h, n, None, None) == want
        assert hkv.hkv_erase(h, n, None) == want
        assert hkv.hkv_insert_and_evict(h, n, None, None, None, ev_keys, None, None,
                                        ev_count) == (INV if dual else want)
        assert hkv.hkv_find_or_insert(h, n, None, None, None, None) == (INV if dual else want)
    torch.cuda.synchronize()
    assert int(ev_count.item()) == 0
    assert t.size() == s0 and t.op_counts() == c0
    for x, y in zip(before, table_state(t)):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    t.close()
