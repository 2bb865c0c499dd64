"""Helpers for the GPU parity tests: move seeded inputs to the device, read
the table back, compare with the oracle."""
import numpy as np
import torch

import workloads as wl

DEV = torch.device("cuda", 0)


def dkeys(a):
    """uint64 numpy -> int64 cuda tensor (same bits)."""
    return torch.from_numpy(wl.as_i64(np.asarray(a, np.uint64))).to(DEV)


def dvals(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(DEV)


def u64(t):
    return t.cpu().numpy().view(np.uint64)


def table_state(t, slot_begin=0, slot_end=None, min_score=0):
    k, v, s = t.export(slot_begin, slot_end, min_score)
    torch.cuda.synchronize()
    return u64(k), v.cpu().numpy(), u64(s)


def assert_same_state(t, o, b_begin=0, b_end=None):
    """Bit-exact: the GPU table's entries of buckets [b_begin, b_end) equal the
    oracle's (keys, values, scores), both sorted by key."""
    b_end = t.num_buckets if b_end is None else b_end
    gk, gv, gs = table_state(t, b_begin * 128, b_end * 128)
    ok, ov, os_ = o.export(b_begin, b_end)
    assert gk.size == ok.size, (gk.size, ok.size)
    assert np.array_equal(gk, ok), "keys differ"
    assert np.array_equal(gs, os_), "scores differ"
    assert np.array_equal(gv.view(np.uint32), ov.view(np.uint32)), "values differ"


def find_compare(t, o, q):
    """find on both sides: found flags, values and scores bit-exact; the value
    and score rows of misses keep their prefilled pattern on both sides.
    Returns the number of hits."""
    n = q.size
    pre = np.full((n, o.dim), -7.25, np.float32)
    pre_s = np.full(n, 0xABCDEF, np.uint64)
    gv, gf, gs = t.find(dkeys(q), values_out=dvals(pre), scores_out=dkeys(pre_s))
    torch.cuda.synchronize()
    ov, of, os_ = o.find(q, values_out=pre.copy(), scores_out=pre_s.copy())
    gf = gf.cpu().numpy()
    assert np.array_equal(gf, of), f"found differs at {np.flatnonzero(gf != of)[:5]}"
    assert np.array_equal(gv.cpu().numpy().view(np.uint32), ov.view(np.uint32)), "values differ"
    assert np.array_equal(u64(gs), os_), "scores differ"
    return int(of.sum())


def read_device(addr, nbytes):
    """Copy nbytes at a raw device address to a numpy byte array (CUDA runtime
    already loaded by torch)."""
    import ctypes
    rt = ctypes.CDLL("libcudart.so.13")
    buf = np.empty(nbytes, np.uint8)
    err = rt.cudaMemcpy(ctypes.c_void_p(buf.ctypes.data), ctypes.c_void_p(int(addr)),
                        ctypes.c_size_t(nbytes), ctypes.c_int(2))
    assert err == 0, err
    return buf
