"""Pins for the oracle's score policies (HKV §3.3 "Scoring policies" and
§5 Exp #3c / Table 8 name kLru, kLfu, kEpochLru, kEpochLfu and kCustomized;
the update rules are the oracle's reading R10).  CPU only.

What pins them, other than the oracle itself:
* kLru and kEpochLru reduce to kCustomized with an explicit score per call
  (the call's clock), a path the main pins already fix;
* kLfu and kEpochLfu: the brute-force model of ``tests/brute.py`` and the
  closed form "score = number of presentations" while no key is displaced;
* saturation at 2^64 - 1 and 2^32 - 1 on hand-picked increments;
* Table 8's shape: frequency-based admission beats recency on a skewed
  stream, and the policies converge once the hot set fits.
"""
import numpy as np
import pytest

import workloads as wl
from tests.brute import BruteTable

MASK = (1 << 64) - 1
LOW32 = (1 << 32) - 1


def _state(t):
    k, v, s = t.export()
    return k, v, s


def _same(a, b):
    for x, y in zip(_state(a), _state(b)):
        assert np.array_equal(x, y)


def _brute_same(o, br):
    ok, ov, os_ = o.export()
    bk, bv, bs = br.export()
    assert np.array_equal(ok, bk)
    assert np.array_equal(os_, bs)
    assert np.array_equal(ov, bv)


def _ops(seed, universe, n_calls, batch, dim):
    """A seeded mix of insert_or_assign / insert_and_evict / find_or_insert /
    assign / erase calls over a small key universe (duplicates included)."""
    rng = np.random.default_rng(seed)
    ops = []
    for c in range(n_calls):
        kind = rng.choice(["ioa", "ioa", "ioa", "iae", "foi", "assign", "erase"])
        k = universe[rng.integers(0, universe.size, batch)]
        v = wl.key_values(k, dim, salt=seed * 1000 + c)
        ops.append((kind, k, v))
    return ops


def _apply(t, kind, k, v, scores=None):
    if kind == "ioa":
        return t.insert_or_assign(k, v, scores)
    if kind == "iae":
        c, ev = t.insert_and_evict(k, v, scores)
        return c, ev
    if kind == "foi":
        c, vals, found = t.find_or_insert(k, v, scores)
        return c, vals, found
    if kind == "assign":
        return t.assign(k, v, scores)
    return t.erase(k)


def _same_result(a, b):
    if isinstance(a, dict):
        assert a == b
        return
    assert a[0] == b[0]
    for x, y in zip(a[1:], b[1:]):
        if isinstance(x, tuple):
            for xx, yy in zip(x, y):
                assert np.array_equal(xx, yy)
        else:
            assert np.array_equal(x, y)


@pytest.mark.parametrize("dual", [False, True])
@pytest.mark.parametrize("epoch", [False, True])
def test_lru_is_customized_with_the_call_clock(oracle_mod, dual, epoch):
    """kLru: every score written by the c-th score-writing call equals c (the
    clock starts at 1); kEpochLru: (epoch << 32) | c.  Replaying the calls on a
    kCustomized table with those scores given explicitly must give the same
    results after every call, in both modes."""
    B, dim = 4, 2
    pol = oracle_mod.POLICY_EPOCH_LRU if epoch else oracle_mod.POLICY_LRU
    a = oracle_mod.OracleTable(B, dim, dual=dual, policy=pol)
    b = oracle_mod.OracleTable(B, dim, dual=dual)
    universe = wl.unique_keys(11, 5 * B * 128)
    clock = 1
    for c, (kind, k, v) in enumerate(_ops(12, universe, 40, 300, dim)):
        if dual and kind in ("iae", "foi"):
            kind = "ioa"
        ep = (7 + c // 5) if epoch else 0
        a.set_epoch(ep)
        want = None
        if kind != "erase":
            want = np.full(k.size, (ep << 32) | clock, np.uint64)
            clock += 1
        _same_result(_apply(a, kind, k, v), _apply(b, kind, k, v, want))
        _same(a, b)
    assert a.step == clock
    with pytest.raises(ValueError):
        a.insert_or_assign(universe[:2], np.zeros((2, dim), np.float32), np.ones(2, np.uint64))


@pytest.mark.parametrize("dual", [False, True])
@pytest.mark.parametrize("policy", ["lfu", "epoch_lfu", "lru", "epoch_lru", "customized"])
def test_policies_match_brute_force(oracle_mod, dual, policy):
    """Every policy, both modes: the oracle equals the independent brute-force
    model after each call of a random stream with in-batch duplicates, caller
    increments (LFU kinds) and epoch changes."""
    import tests.brute as br
    code = {"customized": 0, "lru": 1, "lfu": 2, "epoch_lru": 3, "epoch_lfu": 4}[policy]
    B, dim = 3, 2
    o = oracle_mod.OracleTable(B, dim, dual=dual, policy=code)
    t = BruteTable(B, dim, dual=dual, policy=code)
    universe = wl.unique_keys(21, 4 * B * 128)
    rng = np.random.default_rng(22)
    for c in range(30):
        n = int(rng.integers(1, 400))
        k = universe[rng.integers(0, universe.size, n)]
        v = wl.key_values(k, dim, salt=c)
        scores = None
        if code in (br.LFU, br.EPOCH_LFU, br.CUSTOMIZED) and c % 3:
            scores = rng.integers(0, 5, n).astype(np.uint64)
        if c % 7 == 6:
            o.set_epoch(c)
            t.epoch = c
        if c % 5 == 4:
            co = o.assign(k, v, scores)
            t.assign(k, v, scores)
        else:
            co = o.insert_or_assign(k, v, scores)
            ct = t.insert_or_assign(k, v, scores)
            for f in ("updated", "admitted", "rejected", "evicted", "reserved"):
                assert co[f] == ct[f], f
        _brute_same(o, t)


@pytest.mark.parametrize("policy", ["lfu", "epoch_lfu"])
def test_lfu_score_counts_presentations(oracle_mod, policy):
    """Closed form while nothing is displaced: a key's LFU score is the number
    of times it was presented (every occurrence in every batch, insert_or_assign
    and assign alike); under kEpochLfu the low 32 bits hold that count and the
    high 32 bits the epoch of the last call that presented it."""
    epoch_kind = policy == "epoch_lfu"
    code = oracle_mod.POLICY_EPOCH_LFU if epoch_kind else oracle_mod.POLICY_LFU
    B, dim = 64, 1
    o = oracle_mod.OracleTable(B, dim, policy=code)
    universe = wl.unique_keys(31, 2000)   # far below the 8192 slots: no bucket fills
    rng = np.random.default_rng(32)
    count, last_epoch = {}, {}
    for c in range(25):
        k = universe[rng.integers(0, universe.size, 700)]
        o.set_epoch(100 + c)
        if c % 4 == 3:   # assign presents only resident keys
            o.assign(k, np.zeros(k.size, np.float32))
            pres = [x for x in k.tolist() if x in count]
        else:
            o.insert_or_assign(k, np.zeros(k.size, np.float32))
            pres = k.tolist()
        for x in pres:
            count[x] = count.get(x, 0) + 1
            last_epoch[x] = 100 + c
    keys, _, scores = o.export()
    assert keys.size == len(count)
    for x, s in zip(keys.tolist(), scores.tolist()):
        want = (last_epoch[x] << 32) | count[x] if epoch_kind else count[x]
        assert s == want, (x, s, want)


def test_lfu_saturates(oracle_mod):
    """kLfu adds saturate at 2^64 - 1; kEpochLfu's count at 2^32 - 1 while the
    epoch field is rewritten."""
    k = np.array([5, 5, 9], np.uint64)
    v = np.zeros(3, np.float32)
    o = oracle_mod.OracleTable(1, 1, policy=oracle_mod.POLICY_LFU)
    o.insert_or_assign(k, v, np.array([1 << 63, 1 << 63, MASK - 1], np.uint64))
    o.insert_or_assign(k[2:], v[2:], np.array([3], np.uint64))
    keys, _, s = o.export()
    assert keys.tolist() == [5, 9] and s.tolist() == [MASK, MASK]
    e = oracle_mod.OracleTable(1, 1, policy=oracle_mod.POLICY_EPOCH_LFU)
    e.set_epoch(3)
    e.insert_or_assign(k, v, np.array([1 << 31, 1 << 31, 1], np.uint64))
    e.set_epoch(0xFFFFFFFF)
    e.insert_or_assign(k[2:], v[2:], np.array([LOW32], np.uint64))
    keys, _, s = e.export()
    assert s.tolist() == [(3 << 32) | LOW32, (LOW32 << 32) | LOW32]


def test_lfu_admission_prefers_frequency(oracle_mod):
    """A full bucket of keys seen three times each keeps them against a burst
    of new keys seen once (admission control, HKV Algorithm 2, under kLfu),
    while kLru admits the newer burst."""
    B = 1
    res = wl.unique_keys(41, 128)
    new = wl.unique_keys(42, 64)
    v = np.zeros(128, np.float32)
    lfu = oracle_mod.OracleTable(B, 1, policy=oracle_mod.POLICY_LFU)
    lru = oracle_mod.OracleTable(B, 1, policy=oracle_mod.POLICY_LRU)
    for t in (lfu, lru):
        for _ in range(3):
            t.insert_or_assign(res, v)
    c = lfu.insert_or_assign(new, v[:64])
    assert c["rejected"] == 64 and set(lfu.export()[0].tolist()) == set(res.tolist())
    c = lru.insert_or_assign(new, v[:64])
    assert c["admitted"] == 64 and c["evicted"] == 64


def _hit_rate(oracle_mod, policy, alpha, seed=51):
    """Fraction of lookups found during steady ingestion of a Zipf stream:
    each step finds a batch, then inserts it (the cache workflow of HKV
    Exp #3c), with the epoch advanced once per step."""
    B, batch, steps, warm = 16, 256, 400, 150
    o = oracle_mod.OracleTable(B, 1, policy=policy)
    universe = 32 * B * 128                    # capacity / universe = 1/32
    hits = total = 0
    for step in range(steps):
        k = wl.zipf_keys(seed * 1000 + step, batch, alpha, universe)
        o.set_epoch(step)
        _, f, _ = o.find(k)
        if step >= warm:
            hits += int(f.sum())
            total += k.size
        o.insert_or_assign(k, np.zeros(k.size, np.float32))
    return hits / total


@pytest.mark.slow
def test_table8_shape(oracle_mod):
    """Table 8's shape on a small table: at moderate skew kLfu's hit rate is
    well above kLru's, the epoch policies (epoch advanced per step) track
    kLru, and at alpha 1.25 all of them come close together."""
    P = oracle_mod
    for alpha in (0.75, 0.99):
        lru = _hit_rate(P, P.POLICY_LRU, alpha)
        lfu = _hit_rate(P, P.POLICY_LFU, alpha)
        elru = _hit_rate(P, P.POLICY_EPOCH_LRU, alpha)
        elfu = _hit_rate(P, P.POLICY_EPOCH_LFU, alpha)
        assert lfu > lru + 0.015, (alpha, lfu, lru)
        assert abs(elru - lru) < 1e-12
        assert abs(elfu - lru) < 0.01, (alpha, elfu, lru)
    hi = [_hit_rate(P, p, 1.25) for p in (P.POLICY_LRU, P.POLICY_LFU)]
    assert abs(hi[0] - hi[1]) < 0.01 and min(hi) > 0.8, hi
