"""GPU checks of dual-bucket mode (invariants, since placement depends on the
order the GPU processes absent keys), tiered mode (bit-exact against an
HBM-only twin) and reader/updater/inserter ordering across streams (bit-exact
against the oracle's serial replay in host issue order)."""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.gpu_util import DEV, assert_same_state, dkeys, dvals, table_state, u64

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


def _slots_state(t):
    """(keys, scores, bucket of the slot) of every resident entry: one export
    per bucket, so each entry's bucket is known."""
    ks, ss, bs = [], [], []
    for b in range(t.num_buckets):
        kb, _, sb = t.export(b * 128, b * 128 + 128, with_values=False)
        kb = u64(kb)
        ks.append(kb)
        ss.append(u64(sb))
        bs.append(np.full(kb.size, b, np.uint64))
    return np.concatenate(ks), np.concatenate(ss), np.concatenate(bs)


def _check_dual_invariants(t, o, last_score, last_salt, dim, absent_ok=True):
    keys, scores, buckets = _slots_state(t)
    assert np.unique(keys).size == keys.size, "duplicate keys"
    assert np.bincount(buckets.astype(np.int64), minlength=t.num_buckets).max() <= 128
    b1 = o.buckets_of(keys, 0)
    b2 = o.buckets_of(keys, 1)
    assert np.all((buckets == b1) | (buckets == b2)), "key outside its two candidate buckets"
    # every resident entry carries its last presentation
    want_s = np.array([last_score[int(k)] for k in keys], np.uint64)
    assert np.array_equal(scores, want_s)
    vk, vv, _ = t.export()
    torch.cuda.synchronize()
    vk = u64(vk)
    vv = vv.cpu().numpy()
    for salt in np.unique([last_salt[int(k)] for k in vk[:2000]]):
        sel = np.array([last_salt[int(k)] == salt for k in vk])
        assert np.array_equal(vv[sel], wl.key_values(vk[sel], dim, salt=int(salt)))
    # an absent key is outranked: one candidate bucket is full and its
    # lowest rank is above the key's rank (scores never decrease here)
    res = set(keys.tolist())
    full = np.bincount(buckets.astype(np.int64), minlength=t.num_buckets) == 128
    minrank = {}
    for b in np.flatnonzero(full):
        sel = buckets == b
        j = np.lexsort((keys[sel], scores[sel]))[0]
        minrank[int(b)] = (int(scores[sel][j]), int(keys[sel][j]))
    absent = [k for k in last_score if k not in res]
    for k in absent[:20000]:
        r = (last_score[k], k)
        c = [int(o.bucket(k, 0)), int(o.bucket(k, 1))]
        assert any(cb in minrank and minrank[cb] > r for cb in c), (k, r, c)
    return keys.size


def _first_presentation_check(t, o, batch_keys, batch_scores):
    """Keys of the batch just inserted that are absent after it: Algorithm 3
    applied key by key rejects a key only when both candidate buckets are
    full and each one's lowest rank (score, key) is above the key's; with
    ranks that never fall, both stay that way.  Returns (absent keys, keys
    with a candidate bucket that has a free slot, keys not outranked by both
    buckets).  The batch-wise routing (a key placed by the first bucket pass
    and displaced by the second is not routed again) can leave a few of
    each; the counts say how many."""
    keys, scores, buckets = _slots_state(t)
    occ = np.bincount(buckets.astype(np.int64), minlength=t.num_buckets)
    minrank = {}
    for b in np.unique(buckets).tolist():
        sel = buckets == b
        j = np.lexsort((keys[sel], scores[sel]))[0]
        minrank[int(b)] = (int(scores[sel][j]), int(keys[sel][j]))
    res = set(keys.tolist())
    absent = [(int(k), int(sc)) for k, sc in zip(batch_keys, batch_scores) if int(k) not in res]
    free = weak = 0
    for k, sc in absent:
        cands = [int(o.bucket(k, 0)), int(o.bucket(k, 1))]
        if any(occ[c] < 128 for c in cands):
            free += 1
        if not all(occ[c] == 128 and minrank[c] > (sc, k) for c in cands):
            weak += 1
    return len(absent), free, weak


def test_dual_bucket_invariants(hkv, oracle_mod):
    """Dual mode (HKV Algorithm 3): 1.5 x capacity unique keys with unique
    random scores in batches, then an update batch raising scores; invariants
    after every batch, find consistent with the table, and the retention of
    the top-N scores reported beside the oracle's."""
    B, dim, bs = 256, 8, 4096
    cap = B * 128
    t = hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_DUAL)
    o = oracle_mod.OracleTable(B, dim, dual=True)
    keys = wl.unique_keys(81, int(1.5 * cap))
    scores = wl.stream(82, keys.size) >> np.uint64(2)
    last_score, last_salt = {}, {}
    tot_absent = tot_free = tot_weak = 0
    for i, lo in enumerate(range(0, keys.size, bs)):
        k, s = keys[lo:lo + bs], scores[lo:lo + bs]
        v = wl.key_values(k, dim, salt=i)
        t.reset_op_counts()
        before = t.size()
        t.insert_or_assign(dkeys(k), dvals(v), dkeys(s))
        o.insert_or_assign(k, v, s)
        for kk, ss in zip(k.tolist(), s.tolist()):
            last_score[kk], last_salt[kk] = ss, i
        c = t.op_counts()
        assert c["admitted"] + c["rejected"] == k.size and c["updated"] == 0
        assert t.size() == before + c["admitted"] - c["evicted"]
        # every key of the batch was absent: admitted = those resident now
        assert c["admitted"] == int(t.contains(dkeys(k)).sum().item())
        na, nfree, nweak = _first_presentation_check(t, o, k, s)
        tot_absent += na
        tot_free += nfree
        tot_weak += nweak
        if i % 4 == 3:
            _check_dual_invariants(t, o, last_score, last_salt, dim)
    assert t.error_counts()["timeouts"] == 0
    # updates with higher scores and new values
    res = u64(t.export(with_values=False)[0])
    up = res[:: 3]
    new_s = np.array([last_score[int(x)] + 7 for x in up], np.uint64)
    v = wl.key_values(up, dim, salt=999)
    t.reset_op_counts()
    t.insert_or_assign(dkeys(up), dvals(v), dkeys(new_s))
    assert t.op_counts()["updated"] == up.size
    for kk, ss in zip(up.tolist(), new_s.tolist()):
        last_score[kk], last_salt[kk] = ss, 999
    n_res = _check_dual_invariants(t, o, last_score, last_salt, dim)
    # find agrees with the table contents
    ek, ev, es = t.export()
    torch.cuda.synchronize()
    q = np.concatenate([keys, wl.unique_keys(83, 1000)])
    fv, ff, fs = t.find(dkeys(q))
    torch.cuda.synchronize()
    ff = ff.cpu().numpy().astype(bool)
    ek = u64(ek)
    assert ff.sum() == n_res
    pos = {k: i for i, k in enumerate(ek.tolist())}
    idx = np.array([pos[int(x)] for x in q[ff]])
    assert np.array_equal(fv.cpu().numpy()[ff], ev.cpu().numpy()[idx])
    assert np.array_equal(u64(fs)[ff], u64(es)[idx])
    # top-N retention (HKV Table 11), GPU and oracle
    n_top = cap
    top = {k for k, _ in sorted(last_score.items(), key=lambda kv: (kv[1], kv[0]))[-n_top:]}
    gpu_ret = len(top & set(ek.tolist())) / n_top
    ora_ret = len(top & set(o.export()[0].tolist())) / n_top
    print(f"dual top-N retention: gpu {gpu_ret:.4f} oracle {ora_ret:.4f}; keys absent after "
          f"their batch: {tot_absent}, with a free candidate bucket: {tot_free}, not outranked "
          f"by both candidates: {tot_weak}")
    assert gpu_ret > 0.95 and abs(gpu_ret - ora_ret) < 0.02
    # the departures from key-by-key Algorithm 3 stay rare
    assert tot_free <= 0.01 * tot_absent and tot_weak <= 0.01 * tot_absent


@pytest.mark.parametrize("bs", [1, 37, 300])
def test_dual_two_buckets(hkv, oracle_mod, bs):
    """The smallest dual table, B = 2: every key's two candidate buckets are
    the whole table (b2 is always the other bucket).  Batches of one key up
    to more than the table's 256 slots, unique random scores: after every
    batch the counts add up and, every fourth batch and at the end, the
    invariants hold; once both buckets are full no absent key has a free
    candidate bucket."""
    B, dim = 2, 4
    t = hkv.HashTable(B * 128, dim, mode=hkv.HKV_MODE_DUAL)
    o = oracle_mod.OracleTable(B, dim, dual=True)
    keys = wl.unique_keys(85, 1200)
    scores = wl.stream(86, keys.size) >> np.uint64(2)
    last_score, last_salt = {}, {}
    free_departures = 0
    for i, lo in enumerate(range(0, keys.size, bs)):
        k, sc = keys[lo:lo + bs], scores[lo:lo + bs]
        v = wl.key_values(k, dim, salt=i)
        t.reset_op_counts()
        before = t.size()
        t.insert_or_assign(dkeys(k), dvals(v), dkeys(sc))
        for kk, ss in zip(k.tolist(), sc.tolist()):
            last_score[kk], last_salt[kk] = ss, i
        c = t.op_counts()
        assert c["admitted"] + c["rejected"] == k.size and c["updated"] == 0
        assert t.size() == before + c["admitted"] - c["evicted"] <= B * 128
        assert c["admitted"] == int(t.contains(dkeys(k)).sum().item())
        if before == B * 128:
            _, nfree, _ = _first_presentation_check(t, o, k, sc)
            free_departures += nfree
        if i % 4 == 3:
            _check_dual_invariants(t, o, last_score, last_salt, dim)
    assert t.size() == B * 128
    _check_dual_invariants(t, o, last_score, last_salt, dim)
    assert free_departures == 0
    t.close()


@pytest.mark.parametrize("policy", ["custom", "lru"])
def test_dual_counts_mixed_batches(hkv, oracle_mod, policy):
    """Dual mode on a full table with batches that mix resident keys, fresh
    keys and repeats (fresh keys with tied step scores under LRU): the
    per-call counts agree with the table afterwards -- updated = distinct
    resident keys, admitted = distinct fresh keys now resident, admitted +
    rejected = distinct fresh keys, size grows by admitted - evicted -- and
    the invariants hold."""
    B, dim, bs = 384, 4, 6000
    cap = B * 128
    mode = hkv.HKV_MODE_DUAL | (0 if policy == "custom" else hkv.HKV_POLICY_LRU)
    t = hkv.HashTable(cap, dim, mode=mode)
    keys = wl.unique_keys(91, 3 * cap)
    scores = wl.stream(92, keys.size) >> np.uint64(2)
    custom = policy == "custom"
    pos = 0
    while t.size() < cap and pos < cap * 2:
        k = keys[pos:pos + bs]
        t.insert_or_assign(dkeys(k), dvals(wl.key_values(k, dim, salt=1)),
                           dkeys(scores[pos:pos + bs]) if custom else None)
        pos += bs
    rng = np.random.default_rng(93)
    for r in range(6):
        res = u64(t.export(with_values=False)[0])
        fresh = keys[pos:pos + int(0.6 * bs)]
        pos += fresh.size
        old = rng.choice(res, int(0.3 * bs), replace=False)
        batch = np.concatenate([fresh, old])
        batch = np.concatenate([batch, rng.choice(batch, bs - batch.size)])  # repeats
        rng.shuffle(batch)
        sc = wl.stream(94 + r, batch.size) >> np.uint64(2)
        t.reset_op_counts()
        before = t.size()
        t.insert_or_assign(dkeys(batch), dvals(wl.key_values(batch, dim, salt=10 + r)),
                           dkeys(sc) if custom else None)
        c = t.op_counts()
        fresh_u = np.unique(fresh)
        assert c["updated"] == np.unique(old).size
        assert c["admitted"] + c["rejected"] == fresh_u.size
        assert c["admitted"] == int(t.contains(dkeys(fresh_u)).sum().item())
        assert t.size() == before + c["admitted"] - c["evicted"]
        assert c["evicted"] <= c["admitted"]
    assert t.error_counts()["timeouts"] == 0


@pytest.mark.parametrize("dim", [16, 6, 132])
def test_tiered_equals_hbm_only(hkv, oracle_mod, dim):
    """Tiered mode (HKV §3.6): with half of the value rows in mapped host
    memory every result equals an HBM-only twin bit for bit (dim 6 and 132
    take the find kernel's any-width row copy)."""
    B = 512
    cap = B * 128
    budget = (B // 2) * 128 * 4 * dim
    t = hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_TIERED, value_hbm_bytes=budget)
    h = hkv.HashTable(cap, dim)
    assert t.info()["hbm_value_rows"] == cap // 2
    keys = wl.unique_keys(91, 2 * cap)
    for i, lo in enumerate(range(0, keys.size, 16384)):
        k = keys[lo:lo + 16384]
        v = dvals(wl.key_values(k, dim, salt=i))
        for x in (t, h):
            x.insert_or_assign(dkeys(k), v, None)
        if i % 3 == 2:
            a = dkeys(k[::5])
            av = dvals(wl.key_values(k[::5], dim, salt=100 + i))
            for x in (t, h):
                x.assign(a, av, None)
    for x, y in zip(table_state(t), table_state(h)):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    q = dkeys(np.concatenate([keys[::3], wl.unique_keys(92, 5000)]))
    a = t.find(q)
    b = h.find(q)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_tiered_pool_slab_equals_hbm_only(hkv):
    """A host slab larger than HKV_HOST_SLAB_MAPPED_MAX comes from a host-NUMA
    memory pool (2^27 slots of 64 floats with a 4 GiB HBM budget: 28 GiB of
    rows on the host); every result still equals an HBM-only twin bit for
    bit: finds, assign, export of a host-row slot range."""
    cap, dim, n = 1 << 27, 64, 1 << 20
    budget = 4 << 30
    t = hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_TIERED, value_hbm_bytes=budget)
    h = hkv.HashTable(cap, dim)
    info = t.info()
    assert info["hbm_value_rows"] == budget // (4 * dim) and info["host_values_addr"] != 0
    keys = wl.unique_keys(97, 5 * n)
    for i in range(5):
        k = dkeys(keys[i * n:(i + 1) * n])
        v = wl.key_values_torch(k, dim, salt=10 + i)
        for x in (t, h):
            x.insert_or_assign(k, v, None)
    a = dkeys(keys[::7])
    av = wl.key_values_torch(a, dim, salt=50)
    for x in (t, h):
        x.assign(a, av, None)
    for lo in range(0, keys.size, n):
        q = dkeys(np.concatenate([keys[lo:lo + n:2], wl.unique_keys(98 + lo, n // 8)]))
        ra, rb = t.find(q), h.find(q)
        torch.cuda.synchronize()
        for x, y in zip(ra, rb):
            assert torch.equal(x, y)
    lo = 3 << 25  # slots far above the HBM rows
    for x, y in zip(t.export(lo, lo + (1 << 18)), h.export(lo, lo + (1 << 18))):
        assert torch.equal(x, y)
    t.close()
    h.close()


def test_roles_across_streams(hkv, oracle_mod):
    """insert_or_assign, find and assign issued on three streams in a fixed
    host order give exactly the oracle's serial replay in that order (HKV
    §3.5 Table 4: conflicting roles never overlap)."""
    B, dim = 64, 8
    cap = B * 128
    t = hkv.HashTable(cap, dim)
    o = oracle_mod.OracleTable(B, dim)
    s_ins, s_find, s_upd = (torch.cuda.Stream() for _ in range(3))
    universe = wl.unique_keys(95, 3 * cap)
    rng = np.random.default_rng(5)
    plan = []
    for step in range(12):  # inputs first, all on the device before any call
        k = universe[rng.integers(0, universe.size, 4000)]
        v = wl.key_values(k, dim, salt=step)
        q = universe[rng.integers(0, universe.size, 3000)]
        a = universe[rng.integers(0, universe.size, 2000)]
        av = wl.key_values(a, dim, salt=1000 + step)
        out = (torch.full((q.size, dim), -1.0, device=DEV),
               torch.zeros(q.size, dtype=torch.uint8, device=DEV),
               torch.zeros(q.size, dtype=torch.int64, device=DEV))
        plan.append((k, v, dkeys(k), dvals(v), q, dkeys(q), out, a, av, dkeys(a), dvals(av)))
    torch.cuda.synchronize()
    # issue without host synchronisation: only the library's role events
    # order the three streams
    for (k, v, dk, dv, q, dq, out, a, av, da, dav) in plan:
        t.insert_or_assign(dk, dv, None, stream=s_ins)
        t.find(dq, *out, stream=s_find)
        t.assign(da, dav, None, stream=s_upd)
    torch.cuda.synchronize()
    for (k, v, dk, dv, q, dq, out, a, av, da, dav) in plan:
        o.insert_or_assign(k, v, None)
        ov, of, os_ = o.find(q, values_out=np.full((q.size, dim), -1.0, np.float32),
                             scores_out=np.zeros(q.size, np.uint64))
        gv, gf, gs = out
        assert np.array_equal(gf.cpu().numpy(), of)
        assert np.array_equal(gv.cpu().numpy(), ov)
        assert np.array_equal(u64(gs), os_)
        o.assign(a, av, None)
    assert_same_state(t, o)


@pytest.mark.parametrize("with_scores", [True, False])
def test_dual_assign_exact(hkv, with_scores):
    """assign on a full dual table, batches with resident keys, absent keys
    and repeats: placement is untouched (the export slot of every key stays),
    a resident key takes the values (and score, when given) of its last
    occurrence, everything else keeps its bytes, absent keys stay absent."""
    B, dim = 200, 12
    cap = B * 128
    t = hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_DUAL)
    keys = wl.unique_keys(95, 2 * cap)
    scores = wl.stream(96, keys.size) >> np.uint64(2)
    for lo in range(0, keys.size, 5000):
        k = keys[lo:lo + 5000]
        t.insert_or_assign(dkeys(k), dvals(wl.key_values(k, dim, salt=3)), dkeys(scores[lo:lo + 5000]))
    rng = np.random.default_rng(97)

    def state():  # sorted by key (export order is unspecified)
        k, v, s = table_state(t)
        o = np.argsort(k)
        return k[o], v[o], s[o]

    for r in range(4):
        k0, v0, s0 = state()
        pos = {x: i for i, x in enumerate(k0.tolist())}
        slots0 = _slots_state(t)
        absent = np.setdiff1d(keys, k0)
        batch = np.concatenate([rng.choice(k0, 3000), rng.choice(absent, 1000)])
        rng.shuffle(batch)
        vals = rng.standard_normal((batch.size, dim)).astype(np.float32)
        sc = wl.stream(98 + r, batch.size) >> np.uint64(2)
        t.reset_op_counts()
        t.assign(dkeys(batch), dvals(vals), dkeys(sc) if with_scores else None)
        want_v, want_s = v0.copy(), s0.copy()
        for i, x in enumerate(batch.tolist()):  # in batch order: the last occurrence wins
            j = pos.get(x)
            if j is not None:
                want_v[j] = vals[i]
                if with_scores:
                    want_s[j] = sc[i]
        k1, v1, s1 = state()
        assert np.array_equal(k1, k0)
        slots1 = _slots_state(t)  # every key still in the same bucket
        assert np.array_equal(slots1[0], slots0[0]) and np.array_equal(slots1[2], slots0[2])
        assert np.array_equal(v1.view(np.uint32), want_v.view(np.uint32))
        assert np.array_equal(s1, want_s)
        assert t.op_counts()["updated"] == len({x for x in batch.tolist() if x in pos})
        assert int(t.contains(dkeys(absent)).sum().item()) == 0
    t.close()
