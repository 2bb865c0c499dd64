"""Digest ablation (HierarchicalKV §5.4, Table 7): libhkv_nodigest.so is the
library built with a find that skips the 128-byte digest line and compares
the key against every slot of its bucket.  Its results must be exactly those
of the oracle (and so of the digest build): the digest only filters which
keys are compared, it never decides a result.

The ablation library is loaded in a spawned child process (the binding
serves one library per process); the child compares found flags, values and
scores with the oracle bit for bit and reports back."""
import multiprocessing as mp

import pytest

pytestmark = pytest.mark.gpu


def _child(q, cap, dim, seed):
    try:
        import numpy as np
        import torch

        import hash_table_cache_gb300 as hkv
        from hash_table_cache_gb300 import _build
        import oracle
        import workloads as wl
        from tests.gpu_util import dkeys, dvals, find_compare

        lib = hkv.load(_build.NODIGEST_LIB)
        assert lib._name == _build.NODIGEST_LIB
        oracle.build()
        t = hkv.HashTable(cap, dim)
        o = oracle.OracleTable(cap // 128, dim)
        keys = wl.unique_keys(seed, int(1.3 * cap))
        hits = 0
        # fill past capacity in three batches (evictions in the last), then
        # find residents, evicted keys and fresh keys
        for part in np.array_split(keys, 3):
            v = wl.key_values(part, dim, salt=seed)
            sc = wl.stream(seed + 1, part.size) % np.uint64(5000)
            t.insert_or_assign(dkeys(part), dvals(v), dkeys(sc))
            o.insert_or_assign(part, v, sc)
        q_keys = np.concatenate([keys, wl.unique_keys(seed + 2, cap // 2)])
        q_keys = q_keys[wl.permutation(seed + 3, q_keys.size)]
        hits = find_compare(t, o, q_keys)
        assert 0 < hits < q_keys.size
        t.close()
        torch.cuda.synchronize()
        q.put(("ok", hits))
    except BaseException as exc:  # report any failure to the parent
        import traceback
        q.put(("fail", traceback.format_exc()))


@pytest.mark.parametrize("cap,dim,seed", [(64 * 128, 8, 11), (3 * 128, 5, 12), (1024 * 128, 32, 13)])
def test_nodigest_find_equals_oracle(cap, dim, seed):
    from hash_table_cache_gb300 import _build
    _build.build_all()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_child, args=(q, cap, dim, seed))
    p.start()
    status, info = q.get(timeout=600)
    p.join(timeout=60)
    assert status == "ok", info
    assert p.exitcode == 0
