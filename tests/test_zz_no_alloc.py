"""hkv_insert_or_assign_noalloc: insert_or_assign for callers that cannot let
the library allocate device memory (a serving loop that must never enter
cudaMalloc/cudaFree, which can synchronise the device; a process whose device
memory is already owned by a framework's caching allocator; a fixed memory
budget).  Its working memory is a fixed array inside libhkv.so.

The test drives it through the C ABI and checks, on two calls in a row, that
it leaves exactly the same table as hkv_insert_or_assign on a twin table
(bit-exact, the tolerance of every parity test here), and that a batch too
large for the array is refused without touching the table.  This file is
collected last on purpose."""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.gpu_util import dkeys, dvals, table_state, u64

pytestmark = pytest.mark.gpu


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
