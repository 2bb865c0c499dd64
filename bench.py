#!/usr/bin/env python3
"""Benchmark: batched find + insert_or_assign on the cache-semantic GPU hash
table, single-bucket mode, capacity 2^22 slots, dim 32 (float32 values),
batches of 2^20 keys at an 80% hit rate, load factor swept 0.50 -> 1.00.

One step = one insert_or_assign batch (80% resident keys, 20% fresh, scored
by the step counter) followed by one find batch (80% resident, 20% fresh) on
the full table (load factor 1.00).  `value` = keys processed per second over
the timed steps (both batches), in billions (B-KV/s).  Inputs are resident
in HBM; L2 is flushed (256 MiB write) between steps, outside the timed events.

Also reported: the per-load-factor find and upsert throughput, the roofline
of the dominant kernel against the measured HBM peak, the oracle (CPU) on a
bounded sample, end-to-end throughput with host buffers, and SM clocks.

Multi-GPU (torchrun): every rank runs an independent replica on its own GPU
and its own key stream (no collective on the data path); timing is the max
over ranks and `value` sums the keys of all ranks.

`--impl reference` times the CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "find / insert_or_assign B-KV/s vs load factor 0.5–1.0; % of HBM roofline"
CAP, DIM, BATCH, FILL_BATCH, HIT = 1 << 22, 32, 1 << 20, 1 << 16, 0.8
LAMBDAS = (0.5, 0.75, 0.9, 1.0)
WORKLOAD = "single-bucket, capacity 2^22, dim 32 f32, batch 2^20, 80% hits, step scores"


def find_bytes_per_key(dim, hit):
    """Algorithmic bytes of one find (Algorithm 1): key 8, digest line 128,
    expected key confirms 8*(1 + 127/256) on a hit or 8*128/256 on a miss,
    value row read + output row write 2*4*dim, found flag 1, score read +
    write 16 (hits, scores requested)."""
    d = 4 * dim
    return hit * (8 + 128 + 8 * (1 + 127 / 256) + 2 * d + 1 + 16) + (1 - hit) * (8 + 128 + 4 + 1)


def upsert_bytes(n_keys, dim, n_buckets_touched, n_rows_written, with_scores):
    """Algorithmic bytes of one single-bucket insert_or_assign call (HKV
    Algorithm 2, applied bucket by bucket): per key the input key, value row
    and score (8 + 4*dim + 8*with_scores); per touched bucket its 128
    (key, score) pairs read (2 KiB) and its digest line read and written
    (2 x 128 B); per changed slot its (key, score) pair written (16 B) and
    its value row written (4*dim)."""
    d = 4 * dim
    return (n_keys * (8 + d + 8 * with_scores) + n_buckets_touched * (2048 + 256)
            + n_rows_written * (16 + d))


def probe_access_rates(dim):
    """Random-read rates of this GPU (reads/s) for 32-byte sectors, 128-byte
    lines and value rows of 4*dim bytes, measured by libhkv_probe.so over a
    2 GiB buffer (see csrc/access_probe.cu)."""
    import ctypes
    from hash_table_cache_gb300 import _build
    lib = ctypes.CDLL(_build.PROBE_LIB)
    lib.hkv_probe_random_reads.argtypes = [ctypes.c_uint32, ctypes.c_uint64,
                                           ctypes.POINTER(ctypes.c_double)]
    lib.hkv_probe_random_reads.restype = ctypes.c_int
    rates = {}
    for g in sorted({32, 128, 4 * dim}):
        r = ctypes.c_double(0.0)
        st = lib.hkv_probe_random_reads(g, 2 << 30, ctypes.byref(r))
        rates[g] = r.value if st == 0 else None
    return rates


def find_access_floor(n, dim, hit, num_buckets, rates, hbm_gbs):
    """Lower bound on one find batch from the measured random-read rates: per
    key the key/score sectors of the digest matches (1 + 127/256 on a hit,
    128/256 on a miss) and, on a hit, the value row; one digest line per
    touched bucket; the input keys, output rows, scores and flags streamed at
    the copy bandwidth.  The terms are added (no overlap assumed)."""
    import math
    sectors = n * (hit * (1 + 127 / 256) + (1 - hit) * 128 / 256)
    rows = n * hit
    lines = num_buckets * (1 - math.exp(-n / num_buckets))
    seq = n * (8 + hit * (4 * dim + 8) + 1)
    return sectors / rates[32] + rows / rates[4 * dim] + lines / rates[128] + seq / (hbm_gbs * 1e9)


def upsert_access_floor(n, dim, rows_written, buckets_touched, rates, hbm_gbs):
    """Lower bound on one single-bucket insert_or_assign call from the measured
    random-read rates: per written row one random read of the input row, one
    random write of the table row (costed as a read) and one key/score sector
    write; per touched bucket its 2 KiB of key/score pairs and its digest line
    read and written, plus the input keys, streamed at the copy bandwidth."""
    seq = buckets_touched * (2048 + 256) + 8 * n
    return (2 * rows_written / rates[4 * dim] + rows_written / rates[32]
            + seq / (hbm_gbs * 1e9))


# DRAM bytes (read + write) of one launch, from an ncu capture of the timed
# region of `python bench.py --skip-sweep --no-cpu-baseline --steps 3
# --warmup 3` (the mean of its 3 launches, profiles/launches_c2_step.md),
# valid only while the kernel's sources are the ones captured (sha256 prefix
# over the listed files).
NCU_TRAFFIC = {
    "find_kernel": {"bytes": 162563669 + 65430016, "sources": ("find.cu", "common.cuh", "launch.h"),
                    "sha256": "e4780e0d8a6314bd"},
    "upsert_single_kernel": {"bytes": 178632192 + 55387307,
                             "sources": ("upsert.cu", "common.cuh", "launch.h"),
                             "sha256": "cde1413d76b7a85b"},
}


def ncu_traffic(kernel):
    import hashlib
    rec = NCU_TRAFFIC.get(kernel)
    if not rec:
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        with open(os.path.join(ROOT, "hash_table_cache_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return rec["bytes"] if h.hexdigest()[:16] == rec["sha256"] else None


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during timing."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.window = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(),
                                 f"hkv_bench_clocks_{os.getpid()}_{device_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}", "--format=csv,noheader",
                 "-lms", "10"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.5)  # let the sampler start before the timed region
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def mark(self, t0, t1):
        """Wall-clock bounds of the timed region."""
        self.window = (t0, t1)

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2].split()[0]), float(parts[3].split()[0]),
                             [nm for nm, v in zip(names, parts[6:10]) if v.lower() == "active"]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sel = rows
        if self.window:
            a, b = self.window
            sel = [r for r in rows if a - 0.02 <= r[0] <= b + 0.02]
            if not sel:  # region shorter than the sampling period: nearest samples
                mid = (a + b) / 2
                sel = sorted(rows, key=lambda r: abs(r[0] - mid))[:3]
        reasons = sorted({x for r in sel for x in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": reasons, "samples": len(sel)}


def replica_seed_base(rank):
    """Replicas (one per rank) draw disjoint key streams: every seed of rank r
    is offset by 1000 r."""
    return 1000 * rank


def job_time_and_value(total_s, keys_this_rank, world, device=None):
    """Whole-job figures of the replicas: the slowest rank's timed total
    (max over ranks) and keys of all ranks / that time in B-KV/s.  The only
    collectives of the run (the data path has none)."""
    keys_all = float(keys_this_rank)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_s], dtype=torch.float64, device=device)
        k = torch.tensor([keys_all], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(k, op=dist.ReduceOp.SUM)
        total_s, keys_all = float(t.item()), float(k.item())
    return total_s, keys_all / total_s / 1e9


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args):
    import torch
    import torch.distributed as dist

    import hash_table_cache_gb300 as hkv

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    hkv.load()
    seed_base = replica_seed_base(rank)

    def dk(a):
        return torch.from_numpy(wl.as_i64(a)).to(dev)

    def fill(t, target, pos, keys):
        while t.size() < target and pos < keys.size:
            k = keys[pos:pos + FILL_BATCH]
            t.insert_or_assign(dk(k), wl.key_values_torch(dk(k), DIM, salt=1), None)
            pos += FILL_BATCH
        return pos

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def timed(fn):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) * 1e-3

    keys = wl.unique_keys(3 + seed_base, 2 * CAP)
    sweep = {}
    lambdas = () if args.skip_sweep else LAMBDAS
    # load-factor sweep: find on the filling table; upsert on a re-filled table
    t = hkv.HashTable(CAP, DIM, device=local)
    pos = 0
    for lam in lambdas:
        pos = fill(t, lam * CAP, pos, keys)
        res, _, _ = t.export(with_values=False)
        res = res.cpu().numpy().view(np.uint64)
        q, _ = wl.hit_mix(4 + seed_base, res, 5 + seed_base, BATCH, HIT)
        qd = dk(q)
        vout = torch.empty((BATCH, DIM), dtype=torch.float32, device=dev)
        fout = torch.empty(BATCH, dtype=torch.uint8, device=dev)
        sout = torch.empty(BATCH, dtype=torch.int64, device=dev)
        for _ in range(2):
            t.find(qd, vout, fout, sout)
        ft = [timed(lambda: t.find(qd, vout, fout, sout)) for _ in range(5)]
        sweep[lam] = {"lambda_actual": t.size() / CAP, "find_bkvs": BATCH / statistics.median(ft) / 1e9,
                      "find_hit_rate": float(fout.float().mean().item())}
    t.close()
    for lam in lambdas:
        ut = []
        for rep in range(3):
            t = hkv.HashTable(CAP, DIM, device=local)
            fill(t, lam * CAP, 0, keys)
            res, _, _ = t.export(with_values=False)
            res = res.cpu().numpy().view(np.uint64)
            q, _ = wl.hit_mix(6 + seed_base + rep, res, 7 + seed_base + rep, BATCH, HIT)
            qd = dk(q)
            vd = wl.key_values_torch(qd, DIM, salt=2)
            ut.append(timed(lambda: t.insert_or_assign(qd, vd, None)))
            t.close()
        sweep[lam]["upsert_bkvs"] = BATCH / statistics.median(ut) / 1e9

    # headline: steps at load factor 1.0
    t = hkv.HashTable(CAP, DIM, device=local)
    fill(t, CAP, 0, keys)
    res, _, _ = t.export(with_values=False)
    res = res.cpu().numpy().view(np.uint64)
    nsteps = args.warmup + args.steps
    up_k, up_v, fq = [], [], []
    prev = res
    for s in range(nsteps):
        # upsert: 80% drawn from keys resident before this step (the previous
        # step's upsert keys, all resident after it), 20% fresh
        q, _ = wl.hit_mix(100 + s + seed_base, prev, 200 + seed_base, BATCH, HIT, fresh_start=s * BATCH)
        prev = q
        qd = dk(q)
        up_k.append(qd)
        up_v.append(wl.key_values_torch(qd, DIM, salt=3 + s))
        # find: 80% drawn from the keys this step's upsert just wrote (resident
        # after it: they carry the newest score), 20% fresh
        f, _ = wl.hit_mix(300 + s + seed_base, q, 400 + seed_base, BATCH, HIT, fresh_start=s * BATCH)
        fq.append(dk(f))
    vout = torch.empty((BATCH, DIM), dtype=torch.float32, device=dev)
    fout = torch.empty(BATCH, dtype=torch.uint8, device=dev)
    sout = torch.empty(BATCH, dtype=torch.int64, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nsteps)]
    torch.cuda.synchronize()
    for s in range(args.warmup):
        flush.zero_()
        t.insert_or_assign(up_k[s], up_v[s], None)
        t.find(fq[s], vout, fout, sout)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t.reset_op_counts()
    with Clocks(local) as clk:
        w0 = time.time()
        # NVTX range "timed": lets a profiler select the timed launches
        torch.cuda.nvtx.range_push("timed")
        for s in range(args.warmup, nsteps):
            flush.zero_()
            e0, e1, e2 = ev[s]
            e0.record(stream)
            t.insert_or_assign(up_k[s], up_v[s], None)
            e1.record(stream)
            t.find(fq[s], vout, fout, sout)
            e2.record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        clk.mark(w0, time.time())
    if world > 1:
        dist.barrier()
    up_t = [ev[s][0].elapsed_time(ev[s][1]) * 1e-3 for s in range(args.warmup, nsteps)]
    fi_t = [ev[s][1].elapsed_time(ev[s][2]) * 1e-3 for s in range(args.warmup, nsteps)]
    total = sum(up_t) + sum(fi_t)
    counts = t.op_counts()
    total, value = job_time_and_value(total, 2 * BATCH * args.steps, world, dev)

    # roofline: find is one kernel per call, timed exactly by the events
    # around hkv_find; insert_or_assign is a call of two kernels (stage +
    # bucket processing) and is reported as a call
    peak, peak_kind = read_peaks()
    hit_rate = float(fout.float().mean().item())
    f_avg, u_avg = statistics.mean(fi_t), statistics.mean(up_t)
    fb = find_bytes_per_key(DIM, hit_rate) * BATCH
    rows = (counts["updated"] + counts["admitted"]) / args.steps
    ub = upsert_bytes(BATCH, DIM, CAP // 128, rows, False)
    find_roof = {"bound": "hbm", "achieved": fb / f_avg / 1e9, "peak": peak, "unit": "GB/s",
                 "frac": fb / f_avg / 1e9 / peak, "traffic": ncu_traffic("find_kernel"),
                 "kernel": "find_kernel",
                 "bytes_per_launch": fb, "avg_launch_s": f_avg, "peak_kind": peak_kind}
    up_traffic = ncu_traffic("upsert_single_kernel")
    up_roof = {"bound": "hbm", "achieved": ub / u_avg / 1e9, "peak": peak, "unit": "GB/s",
               "frac": ub / u_avg / 1e9 / peak,
               "traffic": None if up_traffic is None else {"upsert_single_kernel": up_traffic},
               "kernel": "insert_or_assign call (stage_kernel + upsert_single_kernel)",
               "bytes_per_launch": ub, "avg_launch_s": u_avg, "peak_kind": peak_kind}
    dominant = find_roof
    try:
        rates = probe_access_rates(DIM)
        ff = find_access_floor(BATCH, DIM, hit_rate, CAP // 128, rates, peak)
        uf = upsert_access_floor(BATCH, DIM, rows, CAP // 128, rates, peak)
        access = {"random_reads_per_s": {f"{g}B": v for g, v in rates.items()},
                  "find": {"floor_s": ff, "measured_s": f_avg, "frac": ff / f_avg},
                  "insert_or_assign": {"floor_s": uf, "measured_s": u_avg, "frac": uf / u_avg},
                  "note": "floor = random sector/row reads at the probed rates + streamed "
                          "bytes at the copy peak"}
    except Exception as exc:  # the probe is a measurement aid; the line stands without it
        access = {"unavailable": str(exc)}

    # The other calls of the API on the same full table, one 2^20-key batch
    # each (median of 3, L2 flushed before each).
    api = {}
    qk, qv = fq[-1], up_v[-1]
    ptr_out = torch.empty(BATCH, dtype=torch.int64, device=dev)
    api["contains_bkvs"] = BATCH / statistics.median(
        [timed(lambda: t.contains(qk)) for _ in range(3)]) / 1e9
    api["find_ptr_bkvs"] = BATCH / statistics.median(
        [timed(lambda: hkv.hkv_find_ptr(t.handle, BATCH, qk, ptr_out, fout, sout)) for _ in range(3)]) / 1e9
    api["assign_bkvs"] = BATCH / statistics.median(
        [timed(lambda: t.assign(qk, qv, None)) for _ in range(3)]) / 1e9
    ek = torch.empty(BATCH, dtype=torch.int64, device=dev)
    ev_ = torch.empty((BATCH, DIM), dtype=torch.float32, device=dev)
    es = torch.empty(BATCH, dtype=torch.int64, device=dev)
    ec = torch.zeros(1, dtype=torch.int64, device=dev)
    api["insert_and_evict_bkvs"] = BATCH / statistics.median(
        [timed(lambda: hkv.hkv_insert_and_evict(t.handle, BATCH, up_k[s], up_v[s], None, ek, ev_, es, ec))
         for s in range(3)]) / 1e9
    fio_v = [qv.clone() for _ in range(3)]
    api["find_or_insert_bkvs"] = BATCH / statistics.median(
        [timed(lambda: t.find_or_insert(up_k[(s + 3) % nsteps], fio_v[s], None)) for s in range(3)]) / 1e9

    # End to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory, runs insert_or_assign + find and
    # copies the find results back.  Copies run on their own streams, double
    # buffered, so step s+1's upload and step s-1's download overlap step s.
    e2e = None
    if rank == 0 or world > 1:
        ne = args.steps
        hk = [up_k[s % nsteps].cpu().pin_memory() for s in range(2)]
        hv = [up_v[s % nsteps].cpu().pin_memory() for s in range(2)]
        hq = [fq[s % nsteps].cpu().pin_memory() for s in range(2)]
        dk_ = [torch.empty_like(up_k[0]) for _ in range(2)]
        dv_ = [torch.empty_like(up_v[0]) for _ in range(2)]
        dq_ = [torch.empty_like(fq[0]) for _ in range(2)]
        ov_ = [torch.empty((BATCH, DIM), dtype=torch.float32, device=dev) for _ in range(2)]
        of_ = [torch.empty(BATCH, dtype=torch.uint8, device=dev) for _ in range(2)]
        os_ = [torch.empty(BATCH, dtype=torch.int64, device=dev) for _ in range(2)]
        hvo = [torch.empty((BATCH, DIM), dtype=torch.float32).pin_memory() for _ in range(2)]
        hfo = [torch.empty(BATCH, dtype=torch.uint8).pin_memory() for _ in range(2)]
        hso = [torch.empty(BATCH, dtype=torch.int64).pin_memory() for _ in range(2)]
        up_s, dn_s = torch.cuda.Stream(), torch.cuda.Stream()
        in_ready = [torch.cuda.Event() for _ in range(ne)]
        done = [torch.cuda.Event() for _ in range(ne)]
        out_read = [torch.cuda.Event() for _ in range(ne)]
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        up_s.wait_event(a)
        for s in range(ne):
            i = s % 2
            with torch.cuda.stream(up_s):
                if s >= 2:
                    up_s.wait_event(done[s - 2])  # buffers i free again
                dk_[i].copy_(hk[i], non_blocking=True)
                dv_[i].copy_(hv[i], non_blocking=True)
                dq_[i].copy_(hq[i], non_blocking=True)
                in_ready[s].record(up_s)
            stream.wait_event(in_ready[s])
            if s >= 2:
                stream.wait_event(out_read[s - 2])  # output buffers i downloaded
            t.insert_or_assign(dk_[i], dv_[i], None)
            t.find(dq_[i], ov_[i], of_[i], os_[i])
            done[s].record(stream)
            with torch.cuda.stream(dn_s):
                dn_s.wait_event(done[s])
                hvo[i].copy_(ov_[i], non_blocking=True)
                hfo[i].copy_(of_[i], non_blocking=True)
                hso[i].copy_(os_[i], non_blocking=True)
                out_read[s].record(dn_s)
        stream.wait_event(out_read[ne - 1])
        b.record(stream)
        b.synchronize()
        e_total = a.elapsed_time(b) * 1e-3
        bi = hk[0].numel() * 8 + hv[0].numel() * 4 + hq[0].numel() * 8
        bo = hvo[0].numel() * 4 + hfo[0].numel() + hso[0].numel() * 8
        # The host link alone: the same uploads and downloads with no table
        # work between them, both directions on their own streams; the best
        # of 3 runs (the link is shared with the machine's other work).
        link_runs = []
        for _ in range(3):
            torch.cuda.synchronize()
            a.record(stream)
            up_s.wait_event(a)
            dn_s.wait_event(a)
            for s in range(ne):
                i = s % 2
                with torch.cuda.stream(up_s):
                    dk_[i].copy_(hk[i], non_blocking=True)
                    dv_[i].copy_(hv[i], non_blocking=True)
                    dq_[i].copy_(hq[i], non_blocking=True)
                with torch.cuda.stream(dn_s):
                    hvo[i].copy_(ov_[i], non_blocking=True)
                    hfo[i].copy_(of_[i], non_blocking=True)
                    hso[i].copy_(os_[i], non_blocking=True)
            for s_ in (up_s, dn_s):
                x = torch.cuda.Event()
                x.record(s_)
                stream.wait_event(x)
            b.record(stream)
            b.synchronize()
            link_runs.append(a.elapsed_time(b) * 1e-3)
        link_total = min(link_runs)
        e2e = {"value": 2 * BATCH * ne * world / e_total / 1e9, "unit": "B-KV/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "steps": ne, "overlap": "uploads and downloads on their own streams, double buffered",
               "link_only_s_per_step": link_total / ne,
               "frac_of_link_bound": link_total / e_total}
    t.close()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "B-KV/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u64 keys/scores, f32 values (copied)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "capacity": CAP, "dim": DIM, "batch": BATCH,
                   "hit_rate": HIT, "load_factor": 1.0, "mode": "single",
                   "l2": "flushed between steps (256 MiB write), flush outside timed events",
                   "parallelism": f"replicas x{world}"},
        "roofline": dominant,
        "roofline_all": {"find": find_roof, "insert_or_assign": up_roof},
        "access_ceiling": access,
        "per_step": {"insert_or_assign_s": statistics.mean(up_t), "find_s": statistics.mean(fi_t),
                     "find_bkvs": BATCH / f_avg / 1e9, "upsert_bkvs": BATCH / u_avg / 1e9,
                     "find_hit_rate": hit_rate, "op_counts": counts},
        "lambda_sweep": {str(k): v for k, v in sweep.items()},
        "api_at_load_factor_1": api,
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clk.summary(),
        # clear_scratch_kernel + stage_kernel + upsert_single_kernel + find_kernel
        "gpu_launches": args.steps * 4,
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# The other workloads (measurement runs; the default line is the one above)
# ---------------------------------------------------------------------------
OTHER = {
    "c1": "single-bucket, capacity 65,536, dim 8, one batch of 65,536 unique keys (score = index), "
          "then a find of 65,536 keys (half inserted)",
    "c3": "single-bucket, capacity 2^26, dim 64, load factor 1.0, steps of insert_or_assign 2^20 "
          "Zipf(1.05) over 2^32 keys (score = step) + find 2^20 from the same Zipf",
    "c4": "dual-bucket, capacity 2^26, dim 128, unique keys with unique random scores in 2^20 batches "
          "(table full after the untimed prefill), + find 2^20 of the inserted keys",
    "c5": "tiered single-bucket, capacity 2^28, dim 64, 32 GiB of values in HBM and 32 GiB in mapped "
          "host memory, load factor 1.0; mixed stream on three CUDA streams: find 60%, assign 20%, "
          "insert_or_assign 20%, batches of 2^20, Zipf(1.1) over 2^34 keys",
}


def run_other(args):
    import torch

    import hash_table_cache_gb300 as hkv

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    hkv.load()
    cfg = args.config
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def dk(a):
        return torch.from_numpy(wl.as_i64(np.asarray(a, np.uint64))).to(dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def prefill(t, dim, seed, batch=1 << 20, scores=False):
        keys = wl.unique_keys(seed, int(1.6 * t.capacity))
        pos = 0
        while t.size() < t.capacity and pos < keys.size:
            k = dk(keys[pos:pos + batch])
            sc = dk(wl.stream(seed + 1, k.numel(), pos) >> np.uint64(2)) if scores else None
            t.insert_or_assign(k, wl.key_values_torch(k, dim, salt=1), sc)
            pos += batch
        torch.cuda.synchronize()
        return keys[:pos]

    nsteps = args.warmup + args.steps
    times, nkeys, launches = [], [], 0

    def mark_timed(s):
        """NVTX range "timed" over the timed steps (for a profiler)."""
        if s == args.warmup:
            torch.cuda.nvtx.range_push("timed")
    if cfg == "c1":
        cap, dim, n = 65536, 8, 65536
        keys = wl.unique_keys(1, n)
        vals = wl.randn_values(0, n, dim, device=dev)
        sc = dk(np.arange(n, dtype=np.uint64))
        q = np.empty(n, np.uint64)
        q[0::2] = keys[0::2]
        q[1::2] = wl.unique_keys(2, n // 2)
        kd, qd = dk(keys), dk(q)
        t = None
        for s in range(nsteps):
            mark_timed(s)
            if t is not None:
                t.close()
            t = hkv.HashTable(cap, dim)
            flush.zero_()
            a, b = ev(), ev()
            a.record(stream)
            t.insert_or_assign(kd, vals, sc)
            t.find(qd)
            b.record(stream)
            b.synchronize()
            if s >= args.warmup:
                times.append(a.elapsed_time(b) * 1e-3)
                nkeys.append(2 * n)
        launches = 4  # clear, stage, bucket, find
    elif cfg == "c3":
        cap, dim, n = 1 << 26, 64, 1 << 20
        t = hkv.HashTable(cap, dim)
        prefill(t, dim, 6)
        z = wl.Zipf(1.05, 1 << 32)
        for s in range(nsteps):
            mark_timed(s)
            u = dk(wl.zipf_keys(7 + s, n, 1.05, 1 << 32))
            f = dk(wl.zipf_keys(10007 + s, n, 1.05, 1 << 32))
            uv = wl.key_values_torch(u, dim, salt=100 + s)
            torch.cuda.synchronize()
            flush.zero_()
            a, b = ev(), ev()
            a.record(stream)
            t.insert_or_assign(u, uv, None)
            t.find(f)
            b.record(stream)
            b.synchronize()
            if s >= args.warmup:
                times.append(a.elapsed_time(b) * 1e-3)
                nkeys.append(2 * n)
        launches = 4  # clear, stage, bucket, find
    elif cfg == "c4":
        cap, dim, n = 1 << 26, 128, 1 << 20
        t = hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_DUAL)
        inserted = prefill(t, dim, 8, scores=True)
        base = inserted.size
        more = wl.unique_keys(9, nsteps * n)
        for s in range(nsteps):
            mark_timed(s)
            u = dk(more[s * n:(s + 1) * n])
            usc = dk(wl.stream(90, n, s * n) >> np.uint64(2))
            f = dk(wl.choice(10 + s, inserted, n))
            uv = wl.key_values_torch(u, dim, salt=200 + s)
            torch.cuda.synchronize()
            flush.zero_()
            a, b = ev(), ev()
            a.record(stream)
            t.insert_or_assign(u, uv, usc)
            t.find(f)
            b.record(stream)
            b.synchronize()
            if s >= args.warmup:
                times.append(a.elapsed_time(b) * 1e-3)
                nkeys.append(2 * n)
        # clear, dedup, route, bucket pass, clear, retry, bucket pass, finish,
        # find
        launches = 9
    elif cfg == "c5":
        cap, dim, n = 1 << 28, 64, 1 << 20
        t = hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_TIERED, value_hbm_bytes=32 << 30)
        prefill(t, dim, 11)
        sf, sa, su = (torch.cuda.Stream() for _ in range(3))
        kinds = ["find", "find", "find", "assign", "upsert"]
        plan = []
        for s in range(nsteps * 5):
            k = dk(wl.zipf_keys(12 + s, n, 1.1, 1 << 34))
            plan.append((kinds[s % 5], k, wl.key_values_torch(k, dim, salt=0)))
        outs = [(torch.empty((n, dim), device=dev), torch.empty(n, dtype=torch.uint8, device=dev))
                for _ in range(3)]
        torch.cuda.synchronize()
        for s in range(nsteps):
            mark_timed(s)
            a, b = ev(), ev()
            flush.zero_()
            a.record(stream)
            for x, (kind, k, v) in enumerate(plan[5 * s:5 * s + 5]):
                if kind == "find":
                    t.find(k, outs[x][0], outs[x][1], None, with_scores=False, stream=sf)
                elif kind == "assign":
                    t.assign(k, v, None, stream=sa)
                else:
                    t.insert_or_assign(k, v, None, stream=su)
            for st_ in (sf, sa, su):
                e = torch.cuda.Event()
                e.record(st_)
                stream.wait_event(e)
            b.record(stream)
            b.synchronize()
            if s >= args.warmup:
                times.append(a.elapsed_time(b) * 1e-3)
                nkeys.append(5 * n)
        # 3 finds; assign: clear, dedup, assign; upsert: clear, stage, bucket
        launches = 3 + 3 + 3
    torch.cuda.nvtx.range_pop()
    counts = t.op_counts()
    total = sum(times)
    line = {
        "metric": METRIC, "value": sum(nkeys) / total / 1e9, "unit": "B-KV/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / len(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u64 keys/scores, f32 values (copied)", "data": "synthetic",
        "config": {"workload": OTHER[cfg], "name": cfg,
                   "l2": "flushed between steps (256 MiB write), flush outside timed events"},
        "op_counts": counts, "gpu_launches": launches * args.steps,
    }
    t.close()
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline, and the --impl reference arm)
# ---------------------------------------------------------------------------
SAMPLE_EVERY = 8  # the oracle simulates every 8th bucket of the table


def oracle_step_rate(seconds_budget, steps=None):
    """Run the oracle on a bounded sample of the same workload: the buckets b
    with b % 8 == 0 of the 2^22-slot table (filled to load factor 1.0 with the
    same key stream), then steps of (insert_or_assign 2^20, find 2^20) at 80%%
    hits restricted to the keys of those buckets.  Returns (keys/s, steps,
    step times, keys per step)."""
    import oracle
    nb = CAP // 128
    o = oracle.OracleTable(nb, DIM)
    o.set_bucket_filter(np.arange(0, nb, SAMPLE_EVERY, dtype=np.uint64))
    keys = wl.unique_keys(3, 2 * CAP)

    def sampled(k):
        return k[o.buckets_of(k) % np.uint64(SAMPLE_EVERY) == 0]

    pos = 0
    while o.size() < CAP // SAMPLE_EVERY and pos < keys.size:
        k = sampled(keys[pos:pos + FILL_BATCH])
        o.insert_or_assign(k, wl.key_values(k, DIM, salt=1), None)
        pos += FILL_BATCH
    res = o.export()[0]
    times, nkeys = [], []
    s = 0
    t_start = time.perf_counter()
    while True:
        # the full batch restricted to the sampled buckets: 1/8 of the hits
        # (drawn from the residents) and the fresh keys that land there
        m = BATCH // SAMPLE_EVERY
        q = np.concatenate([wl.choice(100 + s, res, int(HIT * m)),
                            sampled(wl.unique_keys(200, int((1 - HIT) * BATCH), s * BATCH))])
        q = q[wl.permutation(150 + s, q.size)]
        v = wl.key_values(q, DIM, salt=3 + s)
        f = np.concatenate([wl.choice(300 + s, q, int(HIT * m)),
                            sampled(wl.unique_keys(400, int((1 - HIT) * BATCH), s * BATCH))])
        a = time.perf_counter()
        o.insert_or_assign(q, v, None)
        o.find(f)
        times.append(time.perf_counter() - a)
        nkeys.append(q.size + f.size)
        s += 1
        if steps is not None and s >= steps:
            break
        if steps is None and time.perf_counter() - t_start > seconds_budget:
            break
    return sum(nkeys) / sum(times), len(times), times, nkeys


def cpu_baseline(seconds):
    rate, n, _, nk = oracle_step_rate(seconds)
    return {"value": rate / 1e9, "unit": "B-KV/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} step(s) of insert_or_assign + find restricted to every "
                      f"{SAMPLE_EVERY}th bucket of the 2^22-slot table at load factor 1.0 "
                      f"(~{int(statistics.mean(nk))} keys per step; fill untimed), single-threaded"}


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    rate, n, times, nk = oracle_step_rate(None, steps=args.warmup + args.steps)
    w = args.warmup if len(times) > args.warmup else 0
    timed, tk = times[w:], nk[w:]
    value = sum(tk) / sum(timed) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "B-KV/s", "n_gpus": world, "steps": len(timed),
        "warmup": args.warmup, "ms_per_step": sum(timed) / len(timed) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u64 keys/scores, f32 values (copied)", "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD, "capacity": CAP, "dim": DIM, "batch": BATCH,
                   "hit_rate": HIT, "load_factor": 1.0, "mode": "single",
                   "parallelism": "cpu, 1 thread"},
        "cpu_baseline": {"value": value, "unit": "B-KV/s", "cores": 1, "kind": "oracle",
                         "sample": f"{len(timed)} timed step(s) of insert_or_assign + find "
                                   f"restricted to every {SAMPLE_EVERY}th bucket of the 2^22-slot "
                                   f"table at load factor 1.0 (~{int(statistics.mean(tk))} keys/step)"},
        "e2e": {"value": value, "unit": "B-KV/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# Build variants: the digest ablation (HKV §5.4, Table 7: find with and
# without the digest line) and the pipelined bucket kernel (next bucket staged
# in shared memory by bulk copies), each against the default build
# ---------------------------------------------------------------------------
def run_ablation_child(lib_path, what):
    """Times one build (the library at lib_path) on the 2^22-slot, dim-32
    table with batches of 2^20 keys; prints one JSON object.  what="find":
    find B-KV/s at load factors 0.5 and 1.0 with 0%, 80% and 100% hits.
    what="upsert": insert_or_assign B-KV/s at load factor 1.0 on the headline
    step mix (80% keys of the previous batch, 20% fresh), median of 10."""
    import torch

    import hash_table_cache_gb300 as hkv

    hkv.load(lib_path)
    dev = torch.device("cuda", 0)
    dk = lambda a: torch.from_numpy(wl.as_i64(a)).to(dev)  # noqa: E731
    keys = wl.unique_keys(3, 2 * CAP)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream()

    def timed(fn):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn()
        b.record(st)
        b.synchronize()
        return a.elapsed_time(b) * 1e-3

    t = hkv.HashTable(CAP, DIM)
    pos, out = 0, {}
    vout = torch.empty((BATCH, DIM), dtype=torch.float32, device=dev)
    fo = torch.empty(BATCH, dtype=torch.uint8, device=dev)
    so = torch.empty(BATCH, dtype=torch.int64, device=dev)
    for lam in ((0.5, 1.0) if what == "find" else (1.0,)):
        while t.size() < lam * CAP and pos < keys.size:
            k = dk(keys[pos:pos + FILL_BATCH])
            t.insert_or_assign(k, wl.key_values_torch(k, DIM, salt=1), None)
            pos += FILL_BATCH
        res = t.export(with_values=False)[0].cpu().numpy().view(np.uint64)
        if what == "find":
            for hit in (0.0, 0.8, 1.0):
                q, _ = wl.hit_mix(4, res, 5, BATCH, hit, fresh_start=(1 + int(lam * 4)) << 24)
                qd = dk(q)
                for _ in range(3):
                    t.find(qd, vout, fo, so)
                ts = [timed(lambda: t.find(qd, vout, fo, so)) for _ in range(5)]
                out[f"find lambda={lam} hits={hit}"] = BATCH / statistics.median(ts) / 1e9
        else:
            batches, prev = [], res
            for r in range(13):
                q, _ = wl.hit_mix(100 + r, prev, 200, BATCH, HIT, fresh_start=r * BATCH)
                prev = q
                qd = dk(q)
                batches.append((qd, wl.key_values_torch(qd, DIM, salt=3 + r)))
            torch.cuda.synchronize()
            ts = [timed(lambda: t.insert_or_assign(k, v, None)) for k, v in batches]
            out["insert_or_assign lambda=1.0"] = BATCH / statistics.median(ts[3:]) / 1e9
    t.close()
    print(json.dumps(out))


def run_ablation(args):
    from hash_table_cache_gb300 import _build
    variant, what = {"digest": ("nodigest", "find"), "pipeline": ("pipeline", "upsert")}[args.ablation]
    res = {}
    for name, lib in (("default_build", _build.LIB), (variant + "_build", _build.VARIANTS[variant][0])):
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--ablation-child", lib,
                            "--ablation-what", what], capture_output=True, text=True, check=True)
        res[name] = json.loads(r.stdout.strip().splitlines()[-1])
    a, b = res["default_build"], res[variant + "_build"]
    print(json.dumps({"ablation": args.ablation, "unit": "B-KV/s",
                      "config": {"workload": "single-bucket, capacity 2^22, dim 32 f32, batch 2^20",
                                 "l2": "flushed before each timed call"},
                      **res, "default_over_variant": {k: a[k] / b[k] for k in a}}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--skip-sweep", action="store_true", help="only the headline steps")
    ap.add_argument("--config", default="c2", choices=["c1", "c2", "c3", "c4", "c5"],
                    help="workload; c2 (the default) is the headline line")
    ap.add_argument("--ablation", choices=["digest", "pipeline"],
                    help="compare the default build with a variant build instead: find without "
                         "the digest line, or the pipelined bucket kernel")
    ap.add_argument("--ablation-child", help=argparse.SUPPRESS)
    ap.add_argument("--ablation-what", default="find", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.ablation_child:
        run_ablation_child(args.ablation_child, args.ablation_what)
    elif args.ablation:
        run_ablation(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.config != "c2":
        run_other(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
