"""GPU parity of the score policies (HKV §3.3 "Scoring policies"; Table 8
names kLru, kLfu, kEpochLru, kEpochLfu, kCustomized; update rules as the
oracle's reading R10).  Single mode is compared with the oracle bit for bit
after every call; dual mode, whose placement depends on the GPU's processing
order, by invariants and by the closed form of LFU counts while no key is
displaced."""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.gpu_util import assert_same_state, dkeys, dvals, find_compare, table_state, u64

pytestmark = pytest.mark.gpu

POLICIES = ["customized", "lru", "lfu", "epoch_lru", "epoch_lfu"]


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


def _codes(hkv, oracle_mod, name):
    lib = {"customized": hkv.HKV_POLICY_CUSTOMIZED, "lru": hkv.HKV_POLICY_LRU,
           "lfu": hkv.HKV_POLICY_LFU, "epoch_lru": hkv.HKV_POLICY_EPOCH_LRU,
           "epoch_lfu": hkv.HKV_POLICY_EPOCH_LFU}[name]
    ora = {"customized": oracle_mod.POLICY_CUSTOMIZED, "lru": oracle_mod.POLICY_LRU,
           "lfu": oracle_mod.POLICY_LFU, "epoch_lru": oracle_mod.POLICY_EPOCH_LRU,
           "epoch_lfu": oracle_mod.POLICY_EPOCH_LFU}[name]
    return lib, ora


@pytest.mark.parametrize("policy", POLICIES)
@pytest.mark.parametrize("num_buckets,dim,max_batch", [(7, 5, 3000), (64, 8, 20000), (8, 4, 12000)])
def test_single_mode_policy_parity(hkv, oracle_mod, policy, num_buckets, dim, max_batch):
    """A seeded stream of insert_or_assign (sparse and dense batches, long
    per-bucket runs with (8, 4)), assign, insert_and_evict, find_or_insert
    and erase calls with duplicates, caller increments and epoch changes:
    table state, counts and outputs equal the oracle's after every call."""
    lib_code, ora_code = _codes(hkv, oracle_mod, policy)
    cap = num_buckets * 128
    t = hkv.HashTable(cap, dim, mode=lib_code)
    o = oracle_mod.OracleTable(num_buckets, dim, policy=ora_code)
    universe = wl.unique_keys(700 + num_buckets, 3 * cap)
    rng = np.random.default_rng(701)
    takes_scores = policy in ("customized", "lfu", "epoch_lfu")
    for step in range(18):
        n = int(rng.integers(1, max_batch))
        keys = universe[rng.integers(0, universe.size, n)]
        vals = wl.key_values(keys, dim, salt=step)
        scores = None
        if takes_scores and step % 3:
            hi = 4 if policy != "customized" else 1 << 40
            scores = rng.integers(0, hi, n).astype(np.uint64)
        ds = None if scores is None else dkeys(scores)
        if step % 4 == 1:
            t.set_epoch(step * 3)
            o.set_epoch(step * 3)
        kind = step % 6
        t.reset_op_counts()
        if kind in (0, 3):
            t.insert_or_assign(dkeys(keys), dvals(vals), ds)
            c = o.insert_or_assign(keys, vals, scores)
            g = t.op_counts()
            for f in ("updated", "admitted", "evicted", "rejected"):
                assert g[f] == c[f], (f, g[f], c[f])
        elif kind == 1:
            t.assign(dkeys(keys), dvals(vals), ds)
            c = o.assign(keys, vals, scores)
            assert t.op_counts()["updated"] == c["updated"]
        elif kind == 2:
            ek, ev, es = t.insert_and_evict(dkeys(keys), dvals(vals), ds)
            torch.cuda.synchronize()
            _, (ok_, ov, os_) = o.insert_and_evict(keys, vals, scores)
            ek = u64(ek)
            order = np.argsort(ek)
            assert np.array_equal(ek[order], ok_)
            assert np.array_equal(u64(es)[order], os_)
            assert np.array_equal(ev.cpu().numpy()[order].view(np.uint32), ov.view(np.uint32))
        elif kind == 4:
            gv = dvals(vals)
            gf = t.find_or_insert(dkeys(keys), gv, ds)
            torch.cuda.synchronize()
            _, ov, of = o.find_or_insert(keys, vals, scores)
            assert np.array_equal(gf.cpu().numpy(), of)
            assert np.array_equal(gv.cpu().numpy().view(np.uint32), ov.view(np.uint32))
        else:
            e = keys[: max(1, n // 4)]
            t.erase(dkeys(e))
            o.erase(e)
        assert_same_state(t, o)
    find_compare(t, o, universe[::3])
    if policy in ("lru", "epoch_lru"):
        with pytest.raises(Exception):
            t.insert_or_assign(dkeys(universe[:2]), dvals(np.zeros((2, dim))), dkeys(np.ones(2, np.uint64)))
    t.close()


@pytest.mark.parametrize("policy", ["lfu", "epoch_lfu"])
def test_lfu_counts_closed_form_both_modes(hkv, oracle_mod, policy):
    """While no key is displaced, a key's LFU score is the number of times it
    was presented (in every mode, since placement is then irrelevant); the
    EpochLfu score carries the epoch of the last presenting call above it."""
    lib_code, _ = _codes(hkv, oracle_mod, policy)
    epoch_kind = policy == "epoch_lfu"
    for mode in (hkv.HKV_MODE_SINGLE, hkv.HKV_MODE_DUAL):
        B, dim = 256, 4
        t = hkv.HashTable(B * 128, dim, mode=mode | lib_code)
        universe = wl.unique_keys(710, 6000)   # about 23 keys per bucket: nothing fills
        rng = np.random.default_rng(711)
        count, last_epoch = {}, {}
        for c in range(20):
            k = universe[rng.integers(0, universe.size, 9000)]
            t.set_epoch(50 + c)
            v = dvals(np.zeros((k.size, dim), np.float32))
            if c % 5 == 4:
                t.assign(dkeys(k), v, None)
                pres = [x for x in k.tolist() if x in count]
            else:
                t.insert_or_assign(dkeys(k), v, None)
                pres = k.tolist()
            for x in pres:
                count[x] = count.get(x, 0) + 1
                last_epoch[x] = 50 + c
        gk, _, gs = table_state(t)
        assert gk.size == len(count)
        want = np.array([((last_epoch[x] << 32) | count[x]) if epoch_kind else count[x]
                         for x in gk.tolist()], np.uint64)
        assert np.array_equal(gs, want)
        t.close()


@pytest.mark.parametrize("policy", POLICIES)
def test_dual_mode_policy_invariants(hkv, oracle_mod, policy):
    """Dual mode under each policy, 2x capacity of keys in batches with
    duplicates: no duplicate keys, every key in one of its two buckets, at
    most 128 per bucket, and each resident key's score is the policy's value
    for its presentations since it was last admitted -- for the clock
    policies the clock of its last presenting call."""
    lib_code, ora_code = _codes(hkv, oracle_mod, policy)
    B, dim = 128, 4
    cap = B * 128
    t = hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_DUAL | lib_code)
    o = oracle_mod.OracleTable(B, dim, dual=True)
    universe = wl.unique_keys(720, 2 * cap)
    rng = np.random.default_rng(721)
    clock, last_clock, last_epoch = 1, {}, {}
    for c in range(24):
        k = universe[rng.integers(0, universe.size, 4096)]
        ep = 9 + c // 4
        t.set_epoch(ep)
        t.insert_or_assign(dkeys(k), dvals(np.zeros((k.size, dim), np.float32)), None)
        for x in k.tolist():
            last_clock[x] = clock
            last_epoch[x] = ep
        clock += 1
    assert t.error_counts()["timeouts"] == 0
    keys, _, scores = table_state(t)
    assert np.unique(keys).size == keys.size
    b1, b2 = o.buckets_of(keys, 0), o.buckets_of(keys, 1)
    # the bucket of each entry, from one export per bucket
    per = np.zeros(B, np.int64)
    for b in range(B):
        kb, _, _ = table_state(t, b * 128, b * 128 + 128)
        per[b] = kb.size
        sel = np.isin(keys, kb)
        assert np.all((b1[sel] == b) | (b2[sel] == b))
    assert per.max() <= 128 and per.sum() == keys.size
    lc = np.array([last_clock[x] for x in keys.tolist()], np.uint64)
    le = np.array([last_epoch[x] for x in keys.tolist()], np.uint64)
    if policy in ("lru", "customized"):
        assert np.array_equal(scores, lc)
    elif policy == "epoch_lru":
        assert np.array_equal(scores, (le << np.uint64(32)) | lc)
    elif policy == "lfu":
        assert np.all(scores >= 1) and np.all(scores <= 24 * 4096)
    else:
        assert np.array_equal(scores >> np.uint64(32), le)
        assert np.all((scores & np.uint64(0xFFFFFFFF)) >= 1)
    t.close()


@pytest.mark.parametrize("policy", POLICIES)
def test_zipf_ingestion_hits_equal_oracle(hkv, oracle_mod, policy):
    """The policy sweep's procedure (HKV §5.4 Exp #3c) at a small scale: a
    2^14-slot table takes batches of Zipf(0.99) keys over 2^19, each looked
    up (contains) and then inserted with the policy's score (customized: the
    step; epoch policies: a new epoch every step).  Every batch's hit count
    and the table after it equal the oracle's, so the sweep's hit rates come
    from the table evolution Algorithm 2 defines."""
    lib_code, ora_code = _codes(hkv, oracle_mod, policy)
    B, dim, n = 128, 4, 1 << 12
    t = hkv.HashTable(B * 128, dim, mode=lib_code)
    o = oracle_mod.OracleTable(B, dim, policy=ora_code)
    zeros = np.zeros((n, dim), np.float32)
    hits = []
    for step in range(1, 13):
        k = wl.zipf_keys(300 + step, n, 0.99, 1 << 19)
        if policy.startswith("epoch"):
            t.set_epoch(step)
            o.set_epoch(step)
        sc = np.full(n, step, np.uint64) if policy == "customized" else None
        g = int(t.contains(dkeys(k)).sum().item())
        _, of, _ = o.find(k)
        assert g == int(of.sum()), (step, g, int(of.sum()))
        hits.append(g)
        t.insert_or_assign(dkeys(k), dvals(zeros), None if sc is None else dkeys(sc))
        o.insert_or_assign(k, zeros, sc)
        assert_same_state(t, o)
    assert hits[-1] > hits[1] > 0  # the hot keys settle in
    t.close()


def test_lfu_increment_sums_saturate(hkv, oracle_mod):
    """LFU increments summed per key within a call, and added to a resident
    key's score, saturate at 2^64 - 1 (the policy's add): one key repeated
    with increments of 2^63 and 2^63 - 1 in one batch, then more in later
    calls, gives the oracle's scores bit for bit."""
    lib_code, ora_code = _codes(hkv, oracle_mod, "lfu")
    B, dim = 4, 2
    t = hkv.HashTable(B * 128, dim, mode=lib_code)
    o = oracle_mod.OracleTable(B, dim, policy=ora_code)
    keys = wl.unique_keys(720, 64)
    rng = np.random.default_rng(721)
    for step in range(6):
        k = np.concatenate([np.repeat(keys[:3], 40), keys[3 + step * 8:11 + step * 8]])
        big = np.array([1 << 63, (1 << 63) - 1, 1, 0], np.uint64)
        inc = big[rng.integers(0, big.size, k.size)] if step % 2 == 0 else \
            rng.integers(0, 1 << 62, k.size).astype(np.uint64)
        v = wl.key_values(k, dim, salt=step)
        t.insert_or_assign(dkeys(k), dvals(v), dkeys(inc))
        o.insert_or_assign(k, v, inc)
        assert_same_state(t, o)
    _, _, gs = t.find(dkeys(keys[:3]))
    torch.cuda.synchronize()
    assert np.all(u64(gs) == np.uint64(2 ** 64 - 1))
    t.close()
