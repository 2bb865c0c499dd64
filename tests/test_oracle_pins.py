"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself (hand-worked examples, closed forms, brute force, the paper's
special cases and statistics).  CPU only."""
import math
import os

import numpy as np
import pytest

import workloads as wl
from tests.brute import BruteTable, fmix64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MASK = (1 << 64) - 1


# --------------------------------------------------------------------------
# Hash: the paper names it only as a Murmur3 derivative (HKV §3.1/§3.2), so its
# exact values are unpinned; we pin the properties of the chosen finalizer.
# --------------------------------------------------------------------------
def test_hash_fixes_zero(oracle_mod):
    # xor-shifts and multiplications both map 0 to 0.
    assert oracle_mod.hash64(0) == 0


def test_hash_is_the_published_bijection(oracle_mod):
    """Invert the oracle's hash with the inverses of the published MurmurHash3
    finalizer steps; a wrong constant, shift or step order fails."""
    c1, c2 = 0xFF51AFD7ED558CCD, 0xC4CEB9FE1A85EC53
    i1, i2 = pow(c1, -1, 1 << 64), pow(c2, -1, 1 << 64)

    def unshift33(y):  # x ^ (x >> 33) is its own inverse on 64 bits
        return y ^ (y >> 33)

    def inverse(h):
        h = unshift33(h)
        h = (h * i2) & MASK
        h = unshift33(h)
        h = (h * i1) & MASK
        return unshift33(h)

    xs = [int(x) for x in wl.stream(11, 2000)] + [1, 2, 3, 1 << 63, MASK]
    for x in xs:
        assert inverse(oracle_mod.hash64(x)) == x


def test_hash_avalanche(oracle_mod):
    """Flipping any input bit flips every output bit with probability ~1/2."""
    xs = [int(x) for x in wl.stream(12, 600)]
    flips = np.zeros((64, 64))
    for x in xs:
        hx = oracle_mod.hash64(x)
        for i in range(64):
            d = hx ^ oracle_mod.hash64(x ^ (1 << i))
            flips[i] += [(d >> j) & 1 for j in range(64)]
    p = flips / len(xs)
    # binomial(600, 1/2): sd ~ 0.02; 0.12 is > 5 sd
    assert np.abs(p - 0.5).max() < 0.12


def test_brute_hash_matches_oracle(oracle_mod):
    for x in wl.stream(13, 100):
        assert fmix64(int(x)) == oracle_mod.hash64(int(x))


# --------------------------------------------------------------------------
# Hand-worked Algorithm 2 walkthrough (golden fixture).
# --------------------------------------------------------------------------
def _parse_entry(tok):
    k, s, v = tok.split(":")
    return int(k), int(s), float(v)


def _range_entries(spec_range, score_spec):
    a, b = (int(x) for x in spec_range.split(".."))
    mul = int(score_spec.split("=")[1].split("*")[0])
    return [(k, mul * k, float(k)) for k in range(a, b + 1)]


def test_golden_alg2_walkthrough(oracle_mod):
    t = oracle_mod.OracleTable(1, 1)
    final = []
    for line in open(os.path.join(GOLDEN, "alg2_one_bucket_walkthrough.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        op, *rest = line.split()
        if op in ("batch", "batch_range"):
            ents = (_range_entries(rest[0], rest[1]) if op == "batch_range"
                    else [_parse_entry(x) for x in rest])
            got = t.insert_or_assign([e[0] for e in ents], [[e[2]] for e in ents],
                                     [e[1] for e in ents])
        elif op == "expect":
            for kv in rest:
                f, n = kv.split("=")
                assert got[f] == int(n), (line, got)
        elif op == "find":
            key = int(rest[0])
            vals, found, scs = t.find([key])
            if rest[2] == "miss":
                assert found[0] == 0, line
            else:
                s, v = rest[2].split(":")
                assert found[0] == 1 and scs[0] == int(s) and vals[0, 0] == float(v), line
        elif op == "final":
            final += [_parse_entry(x) for x in rest]
        elif op == "final_range":
            final += _range_entries(rest[0], rest[1])
    keys, vals, scs = t.export()
    final.sort()
    assert [int(k) for k in keys] == [e[0] for e in final]
    assert [int(s) for s in scs] == [e[1] for e in final]
    assert [float(v) for v in vals[:, 0]] == [e[2] for e in final]


def test_golden_two_bucket_pool(oracle_mod):
    """Algorithm 3 with B = 2: the table is the top-256 pool (see fixture)."""
    text = open(os.path.join(GOLDEN, "alg3_two_bucket_pool.txt")).read()
    pool = int(text.split("capacity_pool")[1].split()[0])
    for seed in range(4):
        t = oracle_mod.OracleTable(2, 1, dual=True)
        keys = wl.unique_keys(100 + seed, 1500)
        scores = wl.stream(200 + seed, 1500) >> np.uint64(40)  # many ties broken by key
        seen = []
        for lo in range(0, 1500, 100):
            k, s = keys[lo:lo + 100], scores[lo:lo + 100]
            t.insert_or_assign(k, np.zeros((100, 1), np.float32), s)
            seen += list(zip(s.tolist(), k.tolist()))
            want = sorted(sorted(seen, reverse=True)[:pool], key=lambda r: r[1])
            got_k, _, got_s = t.export()
            assert got_k.tolist() == [r[1] for r in want]
            assert got_s.tolist() == [r[0] for r in want]
            # phase D1 keeps the two buckets within one entry of each other
            assert abs(t.bucket_size(0) - t.bucket_size(1)) <= 1


# --------------------------------------------------------------------------
# Brute force on tiny tables, random operation mixes.
# --------------------------------------------------------------------------
def _compare(t, ref):
    k1, v1, s1 = t.export()
    k2, v2, s2 = ref.export()
    assert np.array_equal(k1, k2)
    assert np.array_equal(s1, s2)
    assert np.array_equal(v1, v2)


def _random_ops(oracle_mod, dual, seed, num_buckets, dim, steps=30):
    rng = np.random.default_rng(seed)
    t = oracle_mod.OracleTable(num_buckets, dim, dual=dual)
    ref = BruteTable(num_buckets, dim, dual=dual)
    universe = wl.unique_keys(seed + 1000, 3 * 128 * num_buckets)
    for _ in range(steps):
        op = rng.choice(["ioa", "ioa", "ioa", "ioa_step", "assign", "erase", "find"])
        n = int(rng.integers(0, 3 * 128 * num_buckets // 2 + 2))
        keys = universe[rng.integers(0, universe.size, n)]
        if n and rng.random() < 0.3:
            keys[rng.integers(0, n)] = oracle_mod.RESERVED_LO + int(rng.integers(0, 16))
        vals = rng.standard_normal((n, dim)).astype(np.float32)
        scores = rng.integers(0, 40, n).astype(np.uint64)   # small range: many ties
        if op == "ioa":
            c = t.insert_or_assign(keys, vals, scores)
            r = ref.insert_or_assign(keys, vals, scores)
            for f in ("updated", "admitted", "rejected", "evicted", "reserved"):
                assert c[f] == r[f], (f, c, r)
        elif op == "ioa_step":
            c = t.insert_or_assign(keys, vals, None)
            r = ref.insert_or_assign(keys, vals, None)
            for f in ("updated", "admitted", "rejected", "evicted", "reserved"):
                assert c[f] == r[f], (f, c, r)
        elif op == "assign":
            use_s = rng.random() < 0.5
            t.assign(keys, vals, scores if use_s else None)
            ref.assign(keys, vals, scores if use_s else None)
        elif op == "erase":
            t.erase(keys)
            ref.erase(keys)
        else:
            a = t.find(keys)
            b = ref.find(keys)
            for x, y in zip(a, b):
                assert np.array_equal(x, y)
        _compare(t, ref)
        assert t.size() == ref.size()


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("num_buckets,dim", [(1, 1), (2, 3), (3, 4), (5, 2)])
def test_single_bucket_vs_brute(oracle_mod, seed, num_buckets, dim):
    _random_ops(oracle_mod, False, seed, num_buckets, dim)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("num_buckets,dim", [(2, 1), (3, 2), (5, 4)])
def test_dual_bucket_vs_brute(oracle_mod, seed, num_buckets, dim):
    _random_ops(oracle_mod, True, seed, num_buckets, dim)


def test_step_scores(oracle_mod):
    """scores == NULL: one step value per call, +1 per call (DynamicEmb STEP)."""
    t = oracle_mod.OracleTable(4, 1)
    k = wl.unique_keys(5, 10)
    t.insert_or_assign(k[:5], np.zeros((5, 1)), None)
    t.insert_or_assign(k[5:], np.zeros((5, 1)), None)
    t.insert_or_assign(k[:2], np.zeros((2, 1)), None)
    keys, _, scs = t.export()
    want = {int(x): 1 for x in k[:5]} | {int(x): 2 for x in k[5:]} | {int(x): 3 for x in k[:2]}
    assert {int(a): int(b) for a, b in zip(keys, scs)} == want
    assert t.step == 4


def test_alg2_admits_on_equal_score(oracle_mod):
    """HKV Algorithm 2 admits an incoming key whose score equals the bucket
    minimum (score >= min) and evicts the minimum; ties among older entries,
    and among the call's own new entries, go by key.  Hand-worked on one
    bucket (dim 1, value = key)."""
    t = oracle_mod.OracleTable(1, 1)

    def put(keys, score):
        k = np.array(keys, np.uint64)
        return t.insert_or_assign(k, k.astype(np.float32), np.full(k.size, score, np.uint64))

    def keys():
        return sorted(t.export()[0].tolist())

    put(range(1000, 1128), 5)                       # full, every score 5
    c = put([7], 5)                                 # 5 >= 5: admitted, evicts key 1000
    assert c["admitted"] == 1 and c["evicted"] == 1
    assert keys() == [7] + list(range(1001, 1128))
    c = put([3], 4)                                 # 4 < 5: rejected
    assert c["rejected"] == 1 and keys() == [7] + list(range(1001, 1128))
    c = put([9, 2], 5)                              # two new keys; 7 is now old
    assert c["admitted"] == 2 and c["evicted"] == 2
    assert keys() == [2, 9] + list(range(1002, 1128))
    t.erase(np.array([1002], np.uint64))            # one free slot
    c = put([30, 20], 5)                            # free slot, then evicts old key 2
    assert c["admitted"] == 2 and c["evicted"] == 1
    assert keys() == [9, 20, 30] + list(range(1003, 1128))
    # new keys of one call compete by key: 127 entries of score 9, one old
    # entry of score 5, two new keys of score 5 -> the larger new key stays
    t2 = oracle_mod.OracleTable(1, 1)
    k = np.arange(2000, 2127, dtype=np.uint64)
    t2.insert_or_assign(k, k.astype(np.float32), np.full(k.size, 9, np.uint64))
    t2.insert_or_assign(np.array([11], np.uint64), np.ones(1, np.float32), np.array([5], np.uint64))
    c = t2.insert_or_assign(np.array([50, 40], np.uint64), np.ones(2, np.float32),
                            np.array([5, 5], np.uint64))
    assert c["admitted"] == 1 and c["rejected"] == 1 and c["evicted"] == 1
    assert sorted(t2.export()[0].tolist()) == [50] + list(range(2000, 2127))


# --------------------------------------------------------------------------
# Paper special cases and statistics.
# --------------------------------------------------------------------------
def test_table9_admission_burst(oracle_mod):
    """HKV §5.4 Exp #3d / Table 9: a burst scored below every resident is
    fully rejected and changes nothing; a burst scored above every resident is
    fully admitted and displaces exactly the lowest-ranked residents."""
    B = 512
    t = oracle_mod.OracleTable(B, 2)
    keys = wl.unique_keys(21, int(1.6 * B * 128))
    scores = (wl.stream(22, keys.size) % np.uint64(10**9 - 10)) + np.uint64(2)
    for lo in range(0, keys.size, 8192):
        t.insert_or_assign(keys[lo:lo + 8192], np.ones((min(8192, keys.size - lo), 2)),
                           scores[lo:lo + 8192])
    assert t.size() >= 0.96 * B * 128
    before = t.export()
    burst = wl.unique_keys(23, B * 32)
    c = t.insert_or_assign(burst, np.zeros((burst.size, 2)), np.ones(burst.size, np.uint64))
    assert c["admitted"] == 0 and c["rejected"] == burst.size
    after = t.export()
    for x, y in zip(before, after):
        assert np.array_equal(x, y)
    c = t.insert_or_assign(burst, np.zeros((burst.size, 2)),
                           np.full(burst.size, 10**9, np.uint64))
    assert c["admitted"] == burst.size and c["rejected"] == 0
    # per bucket: new contents = top-128 of (old residents + burst keys)
    kb, _, sb = before
    bb = t.buckets_of(kb)
    burst_b = t.buckets_of(burst)
    ka, _, sa = t.export()
    resident_after = set(ka.tolist())
    assert set(burst.tolist()) <= resident_after
    for b in range(0, B, 7):
        old = sorted(zip(sb[bb == b].tolist(), kb[bb == b].tolist()))
        nb = int((burst_b == b).sum())
        drop = max(0, len(old) + nb - 128)
        for rank, (s, k) in enumerate(old):
            assert (k in resident_after) == (rank >= drop)


def _mc_evicted_min(oracle_mod, dual, trials):
    B = 2 if dual else 1
    n = 128 * B
    mins = []
    for tr in range(trials):
        t = oracle_mod.OracleTable(B, 1, dual=dual)
        keys = wl.unique_keys(3000 + tr, n + 1)
        u = wl.stream(4000 + tr, n) >> np.uint64(11)      # 53-bit uniform scores
        t.insert_or_assign(keys[:n], np.zeros((n, 1)), u)
        c = t.insert_or_assign(keys[n:], np.zeros((1, 1)), np.array([1 << 60], np.uint64))
        assert c["evicted"] == 1
        res = set(t.export()[0].tolist())
        victim = [i for i in range(n) if int(keys[i]) not in res]
        assert len(victim) == 1
        mins.append(float(u[victim[0]]) / 2**53)
    return np.mean(mins)


def test_prop33_expected_evicted_score(oracle_mod):
    """HKV Proposition 3.3: with i.i.d. U[0,1] scores in full 128-slot buckets
    the evicted score has mean 1/(n+1) in single mode and 1/(2n+1) when the
    lower of two bucket minima is taken."""
    T = 1500
    single = _mc_evicted_min(oracle_mod, False, T)
    dual = _mc_evicted_min(oracle_mod, True, T)
    # sd of the min of m uniforms ~ 1/(m+1); 5 standard errors
    assert abs(single - 1 / 129) < 5 * (1 / 129) / math.sqrt(T)
    assert abs(dual - 1 / 257) < 5 * (1 / 257) / math.sqrt(T)


def _binom_expected_min128(m, B):
    from scipy.stats import binom
    x = np.arange(0, 129)
    pmf = binom.pmf(x[:-1], m, 1.0 / B)
    return B * (np.sum(x[:-1] * pmf) + 128 * (1 - pmf.sum()))


def test_single_occupancy_closed_form(oracle_mod):
    """Single-bucket mode (HKV §3.2, 128-slot buckets, b = H(k) mod B): after m
    distinct uniform keys with increasing scores, bucket b holds min(128,
    load_b) entries, load_b ~ Binomial(m, 1/B)."""
    B = 2048
    t = oracle_mod.OracleTable(B, 1)
    keys = wl.unique_keys(31, B * 128)
    for i, lo in enumerate(range(0, keys.size, 16384)):
        t.insert_or_assign(keys[lo:lo + 16384], np.zeros((16384, 1)), None)
        m = lo + 16384
        exp = _binom_expected_min128(m, B)
        # sd of the total <= sqrt(B * var(min(128, X))) < sqrt(B * 128)
        assert abs(t.size() - exp) < 5 * math.sqrt(B * 128), (m, t.size(), exp)


def test_first_eviction_load_factor(oracle_mod):
    """HKV §3.4 / Table 11: first eviction near lambda 0.63-0.66 in single mode
    and above 0.97 in dual mode (two-choice placement)."""
    B = 4096
    res = {}
    for dual in (False, True):
        t = oracle_mod.OracleTable(B, 1, dual=dual)
        keys = wl.unique_keys(41, B * 128)
        step = 1024
        first = None
        for lo in range(0, keys.size, step):
            c = t.insert_or_assign(keys[lo:lo + step], np.zeros((step, 1)), None)
            if c["evicted"] + c["rejected"] > 0:
                first = lo / (B * 128)
                break
        res[dual] = first
    # single mode: Poisson model median of the first overflow for this B
    from scipy.stats import poisson
    lam = np.linspace(0.3, 1.0, 701)
    p_ok = poisson.cdf(128, 128 * lam) ** B
    med = lam[np.argmin(np.abs(p_ok - 0.5))]
    assert abs(res[False] - med) < 0.06, (res, med)
    assert res[True] > 0.95, res


def test_bucket_filter_matches_full_model(oracle_mod):
    """The sampled-bucket mode (used for full-size parity) gives the same
    bucket contents as the unfiltered model."""
    B = 64
    full = oracle_mod.OracleTable(B, 2)
    part = oracle_mod.OracleTable(B, 2)
    part.set_bucket_filter([3, 17, 40])
    keys = wl.unique_keys(51, 30000)
    sc = wl.stream(52, 30000) % np.uint64(1000)
    vals = np.arange(60000, dtype=np.float32).reshape(30000, 2)
    for lo in range(0, 30000, 5000):
        for tb in (full, part):
            tb.insert_or_assign(keys[lo:lo + 5000], vals[lo:lo + 5000], sc[lo:lo + 5000])
    for b in (3, 17, 40):
        x = full.export(b, b + 1)
        y = part.export(b, b + 1)
        for u, v in zip(x, y):
            assert np.array_equal(u, v)
    assert part.export(0, 3)[0].size == 0


def test_find_is_membership(oracle_mod):
    """Algorithm 1 returns Found exactly for resident keys, with their row."""
    t = oracle_mod.OracleTable(16, 3)
    keys = wl.unique_keys(61, 4000)
    t.insert_or_assign(keys, np.arange(12000, dtype=np.float32).reshape(4000, 3),
                       wl.stream(62, 4000) % np.uint64(50))
    rk, rv, rs = t.export()
    q = np.concatenate([keys, wl.unique_keys(63, 500)])
    vals, found, scs = t.find(q)
    resident = dict(zip(rk.tolist(), range(rk.size)))
    for i, k in enumerate(q.tolist()):
        if k in resident:
            j = resident[k]
            assert found[i] == 1 and scs[i] == rs[j] and np.array_equal(vals[i], rv[j])
        else:
            assert found[i] == 0


# --------------------------------------------------------------------------
# The cache-workflow operations of HKV §4.1 (insert_and_evict,
# find_or_insert) and §3.5 (contains), against the brute-force model.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("num_buckets,dim", [(1, 2), (3, 3), (7, 4)])
def test_cache_workflow_ops_vs_brute(oracle_mod, seed, num_buckets, dim):
    rng = np.random.default_rng(100 + seed)
    t = oracle_mod.OracleTable(num_buckets, dim)
    ref = BruteTable(num_buckets, dim)
    universe = wl.unique_keys(seed + 2000, 3 * 128 * num_buckets)
    for _ in range(25):
        op = rng.choice(["iae", "fio", "ioa", "contains", "erase"])
        n = int(rng.integers(0, 2 * 128 * num_buckets))
        keys = universe[rng.integers(0, universe.size, n)]
        vals = rng.standard_normal((n, dim)).astype(np.float32)
        scores = rng.integers(0, 40, n).astype(np.uint64)
        use_s = rng.random() < 0.7
        s = scores if use_s else None
        if op == "iae":
            c, (ek, ev, es) = t.insert_and_evict(keys, vals, s)
            out = []
            r = ref.insert_or_assign(keys, vals, s, evicted_out=out)
            assert ek.tolist() == [x[0] for x in out]
            assert es.tolist() == [x[1] for x in out]
            assert np.array_equal(ev, np.array([x[2] for x in out], np.float32).reshape(len(out), dim))
            assert c["evicted"] == r["evicted"] == len(out)
        elif op == "fio":
            c, v, f = t.find_or_insert(keys, vals, s)
            rc, rv, rf = ref.find_or_insert(keys, vals, s)
            assert np.array_equal(f, rf) and np.array_equal(v, rv)
            assert c["updated"] == 0
            for fld in ("admitted", "rejected", "evicted"):
                assert c[fld] == rc[fld]
        elif op == "ioa":
            t.insert_or_assign(keys, vals, s)
            ref.insert_or_assign(keys, vals, s)
        elif op == "contains":
            assert np.array_equal(t.contains(keys), ref.find(keys)[1])
        else:
            t.erase(keys)
            ref.erase(keys)
        _compare(t, ref)
