"""The multi-GPU path of the benchmark runs independent replicas (one table
per rank, no collective on the data path); its only collectives combine the
ranks' timings.  Checked here with two `gloo` processes on the CPU: the job
time is the slowest rank's, the value counts every rank's keys, and the
ranks draw disjoint key streams."""
import multiprocessing as mp
import os
import socket

import numpy as np

import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    try:
        import torch.distributed as dist
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import bench
        total, value = bench.job_time_and_value(1.0 + rank, 100 * (rank + 1), world)
        dist.destroy_process_group()
        q.put((rank, total, value))
    except BaseException as exc:  # report to the parent
        q.put((rank, "fail", repr(exc)))


def test_job_time_and_value_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
    for rank, total, value in out:
        assert total == 2.0, (rank, total, value)  # the slower rank's time
        assert abs(value - 300 / 2.0 / 1e9) < 1e-18  # both ranks' keys
    assert all(p.exitcode == 0 for p in ps)


def test_single_rank_needs_no_collective():
    import bench
    assert bench.job_time_and_value(0.5, 10, 1) == (0.5, 10 / 0.5 / 1e9)


def test_replica_key_streams_are_disjoint():
    import bench
    a = wl.unique_keys(3 + bench.replica_seed_base(0), 1 << 16)
    b = wl.unique_keys(3 + bench.replica_seed_base(1), 1 << 16)
    assert np.intersect1d(a, b).size == 0
