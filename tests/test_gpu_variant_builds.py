"""The measurement builds of the library must compute exactly what the
default build computes:

* libhkv_nodigest.so -- the digest ablation (HierarchicalKV §5.4, Table 7):
  find skips the 128-byte digest line and compares the key against every
  slot of its bucket.  The digest only filters which keys are compared; it
  never decides a result.
* libhkv_pipeline.so -- the bucket kernel stages each warp's next bucket in
  shared memory with bulk copies; only the timing of its loads changes.

Each library is loaded in a spawned child process (the binding serves one
library per process); the child runs inserts with evictions, updates and
finds against the oracle, compares the whole table and every find result bit
for bit, and reports back."""
import multiprocessing as mp

import pytest

pytestmark = pytest.mark.gpu


def _child(q, variant, cap, dim, seed):
    try:
        import numpy as np
        import torch

        import hash_table_cache_gb300 as hkv
        from hash_table_cache_gb300 import _build
        import oracle
        import workloads as wl
        from tests.gpu_util import assert_same_state, dkeys, dvals, find_compare

        path = _build.VARIANTS[variant][0]
        lib = hkv.load(path)
        assert lib._name == path
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
            assert_same_state(t, o)
        # a step-scored batch of residents and fresh keys (updates + evictions)
        mix = np.concatenate([keys[::3], wl.unique_keys(seed + 4, cap // 4)])
        v = wl.key_values(mix, dim, salt=seed + 5)
        t.insert_or_assign(dkeys(mix), dvals(v), None)
        o.insert_or_assign(mix, v, None)
        assert_same_state(t, o)
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


@pytest.mark.parametrize("variant", ["nodigest", "pipeline"])
@pytest.mark.parametrize("cap,dim,seed", [(64 * 128, 8, 11), (3 * 128, 5, 12), (1024 * 128, 32, 13)])
def test_variant_build_equals_oracle(variant, cap, dim, seed):
    from hash_table_cache_gb300 import _build
    _build.build_all()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_child, args=(q, variant, cap, dim, seed))
    p.start()
    status, info = q.get(timeout=600)
    p.join(timeout=60)
    assert status == "ok", info
    assert p.exitcode == 0
