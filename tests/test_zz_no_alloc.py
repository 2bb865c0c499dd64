"""hkv_insert_or_assign_noalloc: insert_or_assign for callers that cannot let
the library allocate device memory (a serving loop that must never enter
cudaMalloc/cudaFree, which can synchronise the device; a process whose device
memory is already owned by a framework's caching allocator; a fixed memory
budget).  Its working memory is a fixed array inside libhkv.so.

The tests drive it through the C ABI and check, on two calls in a row, that
it leaves exactly the same table as hkv_insert_or_assign on a twin table
(bit-exact, the tolerance of every parity test here; dual mode, whose
placement depends on processing order, by its invariants and equal outcome
totals), that batches at the array's limit are accepted and one key more is
refused without touching the table, and that the call is ordered on the
table like any inserter.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.gpu_util import dkeys, dvals, table_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="module")
def hkv():
    import hash_table_cache_gb300 as m
    from hash_table_cache_gb300 import _build
    _build.build()
    m.load()
    return m


def _same(a, b):
    ka, va, sa = table_state(a)
    kb, vb, sb = table_state(b)
    assert np.array_equal(ka, kb)
    assert np.array_equal(sa, sb)
    assert np.array_equal(va.view(np.uint32), vb.view(np.uint32))


def test_noalloc_matches_insert_or_assign_twice(hkv):
    """Single-bucket mode, where a batch's result does not depend on GPU
    scheduling, so two tables fed the same calls must match bit for bit."""
    cap, dim = 512 * 128, 8
    ref = hkv.HashTable(cap, dim)
    noa = hkv.HashTable(cap, dim)
    keys1 = wl.unique_keys(901, 60000)
    # second call: half the first call's keys again (updates), fresh keys
    # beyond the free slots (evictions and rejections) and in-batch duplicates
    keys2 = np.concatenate([keys1[::2], wl.unique_keys(902, 40000), keys1[:500]])
    for call, (k, scores) in enumerate([(keys1, wl.stream(903, keys1.size) % np.uint64(1000)),
                                        (keys2, None)]):
        v = wl.key_values(k, dim, salt=call)
        dk, dv = dkeys(k), dvals(v)
        ds = None if scores is None else dkeys(scores)
        assert hkv.hkv_insert_or_assign(ref.handle, k.size, dk, dv, ds) == hkv.HKV_OK
        assert hkv.hkv_insert_or_assign_noalloc(noa.handle, k.size, dk, dv, ds) == hkv.HKV_OK
        torch.cuda.synchronize()
        _same(ref, noa)
        assert ref.size() == noa.size()
        assert ref.op_counts() == noa.op_counts()
    q = dkeys(np.concatenate([keys2, wl.unique_keys(904, 1000)]))
    a = ref.find(q)
    b = noa.find(q)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    ref.close()
    noa.close()


def test_noalloc_refuses_batches_beyond_the_array(hkv):
    t = hkv.HashTable(256 * 128, 4)
    n = 1 << 21  # needs more than the array holds
    k = torch.arange(1, n + 1, dtype=torch.int64, device="cuda")
    v = torch.zeros((n, 4), dtype=torch.float32, device="cuda")
    assert hkv.hkv_insert_or_assign_noalloc(t.handle, n, k, v, None) == hkv.HKV_ERR_INVALID
    assert t.size() == 0
    ok = hkv.hkv_insert_or_assign_noalloc(t.handle, 1000, k, v, None)
    assert ok == hkv.HKV_OK and t.size() == 1000
    t.close()


def test_noalloc_is_ordered_like_an_inserter(hkv):
    """The call records its role event on the table: a find issued on another
    stream right after it sees its keys, and reading the counts or destroying
    the table waits for it, with no synchronisation by the caller."""
    t = hkv.HashTable(1024 * 128, 16)
    k = wl.unique_keys(911, 100000)
    v = wl.key_values(k, 16, salt=5)
    dk, dv = dkeys(k), dvals(v)
    torch.cuda.synchronize()
    s1 = torch.cuda.Stream()
    s2 = torch.cuda.Stream()
    assert hkv.hkv_insert_or_assign_noalloc(t.handle, k.size, dk, dv, None, s1) == hkv.HKV_OK
    vout = torch.empty((k.size, 16), dtype=torch.float32, device="cuda")
    fout = torch.empty(k.size, dtype=torch.uint8, device="cuda")
    assert hkv.hkv_find(t.handle, k.size, dk, vout, fout, None, s2) == hkv.HKV_OK
    counts = t.op_counts()  # waits for the table's recorded calls
    assert counts["admitted"] + counts["rejected"] == k.size
    s2.synchronize()
    found = fout.cpu().numpy().astype(bool)
    assert found.sum() == counts["admitted"]
    assert np.array_equal(vout.cpu().numpy()[found], v[found])
    # a second call on s1, then destroy at once: destroy waits for it
    k2 = wl.unique_keys(912, 50000)
    dk2, dv2 = dkeys(k2), dvals(wl.key_values(k2, 16, salt=6))
    torch.cuda.synchronize()
    assert hkv.hkv_insert_or_assign_noalloc(t.handle, k2.size, dk2, dv2, None, s1) == hkv.HKV_OK
    t.close()
    del dk2, dv2


def test_noalloc_dual_mode(hkv, oracle_mod):
    """Dual-bucket mode (HKV Algorithm 3) with the array's dual-mode carving:
    two calls in a row on a table fed like its pool-backed twin; both keep the
    dual-mode invariants and report the same outcome totals."""
    from tests.test_gpu_modes import _check_dual_invariants
    B, dim = 256, 8
    ref = hkv.HashTable(B * 128, dim, mode=hkv.HKV_MODE_DUAL)
    noa = hkv.HashTable(B * 128, dim, mode=hkv.HKV_MODE_DUAL)
    o = oracle_mod.OracleTable(B, dim, dual=True)
    keys = wl.unique_keys(921, int(1.4 * B * 128))
    scores = wl.stream(922, keys.size) >> np.uint64(2)
    last_score, last_salt = {}, {}
    half = keys.size // 2
    for call, sl in enumerate((slice(0, half), slice(half, keys.size))):
        k, s = keys[sl], scores[sl]
        v = wl.key_values(k, dim, salt=call)
        dk, dv, ds = dkeys(k), dvals(v), dkeys(s)
        assert hkv.hkv_insert_or_assign(ref.handle, k.size, dk, dv, ds) == hkv.HKV_OK
        assert hkv.hkv_insert_or_assign_noalloc(noa.handle, k.size, dk, dv, ds) == hkv.HKV_OK
        for kk, ss in zip(k.tolist(), s.tolist()):
            last_score[kk], last_salt[kk] = ss, call
        torch.cuda.synchronize()
        for t in (ref, noa):
            _check_dual_invariants(t, o, last_score, last_salt, dim)
        assert ref.op_counts() == noa.op_counts()
        assert ref.size() == noa.size()
    ref.close()
    noa.close()


@pytest.mark.parametrize("policy,limit", [("custom", 1 << 20), ("lfu", 1 << 19)])
def test_noalloc_size_limit_both_sides(hkv, policy, limit):
    """The largest batch the array holds is accepted and gives the same table
    as hkv_insert_or_assign; one key more is refused and changes nothing.
    Single mode: 2^20 keys, 2^19 under the LFU policies (their per-key
    increment sums need room too)."""
    mode = hkv.HKV_POLICY_LFU if policy == "lfu" else 0
    cap, dim = 2048 * 128, 4
    ref = hkv.HashTable(cap, dim, mode=mode)
    noa = hkv.HashTable(cap, dim, mode=mode)
    k = wl.unique_keys(931, limit + 1)
    k[-7:] = k[:7]  # a few repeats
    v = wl.key_values(k, dim, salt=1)
    dk, dv = dkeys(k), dvals(v)
    assert hkv.hkv_insert_or_assign_noalloc(noa.handle, limit + 1, dk, dv, None) == hkv.HKV_ERR_INVALID
    assert noa.size() == 0
    assert hkv.hkv_insert_or_assign(ref.handle, limit, dk, dv, None) == hkv.HKV_OK
    assert hkv.hkv_insert_or_assign_noalloc(noa.handle, limit, dk, dv, None) == hkv.HKV_OK
    torch.cuda.synchronize()
    _same(ref, noa)
    assert ref.op_counts() == noa.op_counts()
    ref.close()
    noa.close()


def test_noalloc_dual_size_limit(hkv):
    """Dual mode carves more arrays per key: 2^19 keys fit a small table's
    share of the array, 2^19 + 1 are refused."""
    t = hkv.HashTable(1024 * 128, 4, mode=hkv.HKV_MODE_DUAL)
    n = (1 << 19) + 1
    k = dkeys(wl.unique_keys(941, n))
    v = torch.zeros((n, 4), dtype=torch.float32, device="cuda")
    assert hkv.hkv_insert_or_assign_noalloc(t.handle, n, k, v, None) == hkv.HKV_ERR_INVALID
    assert t.size() == 0
    assert hkv.hkv_insert_or_assign_noalloc(t.handle, n - 1, k, v, None) == hkv.HKV_OK
    assert t.size() > 0
    t.close()
