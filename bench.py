#!/usr/bin/env python3
"""Benchmark: batched find + insert_or_assign on the cache-semantic GPU hash
table, single-bucket mode, capacity 2^22 slots, dim 32 (float32 values),
batches of 2^20 keys at an 80% hit rate, load factor swept 0.50 -> 1.00.

One step = one insert_or_assign batch (80% keys resident before the step,
20% fresh, scored by the step counter) followed by one find batch (80% keys
resident after the insert, drawn uniformly from the whole resident set, 20%
fresh) on the full table (load factor 1.00).  `value` = keys processed per
second over the timed steps (both batches), in billions (B-KV/s).  Inputs
are resident in HBM; L2 is flushed (256 MiB write) between steps, outside the
timed events.

Also reported: find and insert_or_assign per load factor (with the roofline
fraction of each), the roofline of the dominant kernel against the measured
HBM peak, the random-access ceiling of this GPU (probed), the other calls of
the API, the other workloads (65,536-slot one-batch table; 2^26-slot Zipf
stream; 2^26-slot dual-bucket stream with its top-N retention; 2^28-slot
tiered mixed stream with its host-link bound), the oracle (CPU) on a bounded
sample, end-to-end throughput with host buffers, and SM clocks.

Multi-GPU (torchrun): every rank runs an independent replica on its own GPU
and its own key stream (no collective on the data path); timing is the max
over ranks and `value` sums the keys of all ranks.

`--impl reference` times the CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
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


# ---------------------------------------------------------------------------
# Byte models.  Algorithmic bytes per key for each path of the method, at 8-
# byte granularity (the bytes the method itself needs), D = 4*dim:
#   find (HKV Algorithm 1): key 8, digest line 128, key confirms
#     8*(1 + 127/256) on a hit (the true slot and the expected false digest
#     matches of a full bucket) or 8*128/256 on a miss, row read + output row
#     write 2D, found flag 1, score read + write 16 on a hit;
#   dual find (HKV §3.4): a key found in its second bucket, or missed, adds
#     that bucket's line and its false matches (128 + 4);
#   insert_or_assign (HKV Algorithm 2): hit 16 + D + 128 + 12 + D + 8; insert
#     into a free slot 16 + 2D + 128 + 4 + 17; evicting insert 1189 + 2D (the
#     bucket's 1 KiB of scores scanned); rejected 1172; a repeat of a key in
#     the same batch (collapsed) 8 + D;
#   dual insert_or_assign (HKV Algorithm 3): an insert into a free slot reads
#     the second line too (+132); an evicting insert (D2) also scans the
#     second bucket (2345 + 2D); a rejection scans both (1172 + 1156).
# ---------------------------------------------------------------------------
def find_bytes_per_key(dim, hit):
    """Algorithmic bytes of one single-mode find at hit rate `hit`."""
    d = 4 * dim
    return hit * (8 + 128 + 8 * (1 + 127 / 256) + 2 * d + 1 + 16) + (1 - hit) * (8 + 128 + 4 + 1)


def find_bytes_dual(dim, n_first, n_second, n_miss):
    """Algorithmic bytes of one dual-mode find batch: keys found in their
    first bucket, found in their second, not found."""
    d = 4 * dim
    hit = 8 + 128 + 8 * (1 + 127 / 256) + 2 * d + 1 + 16
    return n_first * hit + n_second * (hit + 132) + n_miss * (8 + 128 + 4 + 1 + 132)


def upsert_bytes(n_keys, dim, n_buckets_touched, n_rows_written, with_scores):
    """Bytes of one single-bucket insert_or_assign call under this build's
    slot layout (HKV Algorithm 2 applied bucket by bucket): per key the input
    key, value row and score (8 + 4*dim + 8*with_scores); per touched bucket
    its 128 (key, score) pairs read (2 KiB) and its digest line read and
    written (2 x 128 B); per changed slot its (key, score) pair written (16 B)
    and its value row written (4*dim)."""
    d = 4 * dim
    return (n_keys * (8 + d + 8 * with_scores) + n_buckets_touched * (2048 + 256)
            + n_rows_written * (16 + d))


def upsert_bytes_paths(counts, n_keys, dim, dual=False):
    """Algorithmic bytes of one insert_or_assign call from its outcome
    counts, path by path (see the table above): updated keys take the hit
    path, evicted residents one evicting insert each, the other admitted keys
    an insert into a free slot, rejected keys the reject path, and the keys
    the batch repeats the repeat path."""
    d = 4 * dim
    upd, adm, ev, rej = (counts[k] for k in ("updated", "admitted", "evicted", "rejected"))
    free_ins = max(adm - ev, 0)
    repeats = max(n_keys - upd - adm - rej, 0)
    if dual:
        return (upd * (164 + 2 * d) + free_ins * (165 + 2 * d + 132) + ev * (2345 + 2 * d)
                + rej * (1172 + 1156) + repeats * (8 + d))
    return (upd * (164 + 2 * d) + free_ins * (165 + 2 * d) + ev * (1189 + 2 * d) + rej * 1172
            + repeats * (8 + d))


def assign_bytes_per_hit(dim):
    """Algorithmic bytes of one assign hit (HKV §3.5): input key and row,
    digest line, key confirm, row write, score write."""
    d = 4 * dim
    return 16 + 2 * d + 140


# ---------------------------------------------------------------------------
# Probes of this GPU: random-read rates and the host link (libhkv_probe.so).
# ---------------------------------------------------------------------------
def _probe_lib():
    import ctypes
    from hash_table_cache_gb300 import _build
    lib = ctypes.CDLL(_build.PROBE_LIB)
    lib.hkv_probe_random_reads_at.argtypes = [ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int,
                                              ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    lib.hkv_probe_random_reads_at.restype = ctypes.c_int
    lib.hkv_probe_host_link.argtypes = [ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64,
                                        ctypes.POINTER(ctypes.c_double)]
    lib.hkv_probe_host_link.restype = ctypes.c_int
    return lib


PROBE_DEPTHS = (2, 4, 8)
PROBE_BLOCKS = (4, 8)


def probe_access_rates(granules):
    """Random reads per second of each granule size over a 2 GiB buffer: the
    plateau (the best rate) over reads in flight per thread or tile
    (PROBE_DEPTHS) and blocks per SM (PROBE_BLOCKS), with the whole grid."""
    import ctypes
    lib = _probe_lib()
    out = {}
    for g in sorted(set(granules)):
        grid = {}
        for d in PROBE_DEPTHS:
            for b in PROBE_BLOCKS:
                r = ctypes.c_double(0.0)
                st = lib.hkv_probe_random_reads_at(g, 2 << 30, d, b, ctypes.byref(r))
                grid[f"d{d}_b{b}"] = r.value if st == 0 else None
        ok = [v for v in grid.values() if v]
        out[g] = {"plateau": max(ok) if ok else None, "grid": grid}
    return out


HOST_SLAB_MAPPED_MAX = 16 << 30  # HKV_HOST_SLAB_MAPPED_MAX of include/hkv.h


def slab_kinds(slab_bytes):
    """The probe kinds (random row reads, writes) over the memory a tiered
    table allocates for a host slab of `slab_bytes`: mapped memory up to
    HOST_SLAB_MAPPED_MAX, a host-NUMA pool above."""
    return (2, 3) if slab_bytes <= HOST_SLAB_MAPPED_MAX else (6, 7)


def probe_host_link(row_bytes, buffer_bytes=1 << 30, kinds=(0, 1, 2, 3)):
    """SM loads and stores over pinned host memory allocated as a tiered
    table's slab is (the path tiered rows take): streaming and random rows of
    `row_bytes` over a buffer of `buffer_bytes`, bytes per second."""
    import ctypes
    lib = _probe_lib()
    names = {0: "stream_read", 1: "stream_write", 2: "row_read", 3: "row_write",
             6: "row_read", 7: "row_write"}  # 4 + kind: pool memory
    out = {}
    for kind in kinds:
        r = ctypes.c_double(0.0)
        st = lib.hkv_probe_host_link(kind, row_bytes, buffer_bytes, ctypes.byref(r))
        out[names[kind]] = r.value if st == 0 else None
    return out


def access_floor(random_counts, seq_bytes, rates, hbm_gbs):
    """Lower bound on a launch: each random access at the probed plateau rate
    of its granule, plus the streamed bytes at the copy peak (terms added, no
    overlap assumed).  random_counts = {granule bytes: accesses}."""
    t = seq_bytes / (hbm_gbs * 1e9)
    for g, c in random_counts.items():
        t += c / rates[g]["plateau"]
    return t


def find_random_counts(n, dim, hit, num_buckets, line_dram=1.0):
    """Random accesses of one single-mode find batch: the key/score sectors of
    the candidates (1 + 127/256 on a hit, 128/256 on a miss), one value row
    per hit, one digest line per touched bucket (`line_dram` = share of them
    that reach DRAM)."""
    sectors = n * (hit * (1 + 127 / 256) + (1 - hit) * 128 / 256)
    rows = n * hit
    lines = num_buckets * (1 - math.exp(-n / num_buckets)) * line_dram
    row_g = max(32, 4 * dim) if 4 * dim <= 128 else 4 * dim
    counts = {32: sectors, 128: lines}
    counts[row_g] = counts.get(row_g, 0) + rows
    return counts


# ---------------------------------------------------------------------------
# The table's documented hash (include/hkv.h): H = 64-bit MurmurHash3
# finalizer, b1 = H(k) mod B, b2 = H(k ^ 0x9E3779B97F4A7C15) mod B moved to
# (b1 + 1) mod B when equal.  Used here only to split measured dual-mode hits
# into first- and second-bucket hits for the byte model.
# ---------------------------------------------------------------------------
def _fmix64_t(x):
    import torch

    def shr(v, s):
        return (v >> s) & ((1 << (64 - s)) - 1)
    x = x ^ shr(x, 33)
    x = x * wl._i64(0xff51afd7ed558ccd)
    x = x ^ shr(x, 33)
    x = x * wl._i64(0xc4ceb9fe1a85ec53)
    return x ^ shr(x, 33)


def first_bucket_t(keys, num_buckets):
    """b1 of int64 key tensors for a power-of-two bucket count."""
    return _fmix64_t(keys) & (num_buckets - 1)


def second_bucket_t(keys, b1, num_buckets):
    b2 = _fmix64_t(keys ^ wl._i64(0x9E3779B97F4A7C15)) & (num_buckets - 1)
    return b2 + (b2 == b1).to(b2.dtype) * (((b1 + 1) % num_buckets) - b2)


def rows_of_ptrs(ptrs, found, info):
    """Row index of each found key from find* row addresses (hkv_info)."""
    import torch
    rb = 4 * info["dim"]
    p = ptrs.clone()
    hbm = info["hbm_values_addr"]
    rows = torch.where(found.bool(), (p - hbm) // rb, torch.zeros_like(p))
    if info["host_values_addr"]:
        host = info["host_values_addr"]
        in_host = found.bool() & ((p < hbm) | (p >= hbm + info["hbm_value_rows"] * rb))
        rows = torch.where(in_host, info["hbm_value_rows"] + (p - host) // rb, rows)
    return rows


# ---------------------------------------------------------------------------
# DRAM bytes (read + write) of one launch from an ncu capture, valid only
# while the kernel's sources are the ones captured (sha256 prefix over the
# listed files); null otherwise.  Captured from the timed region of
# `python bench.py --skip-sweep --skip-configs --no-cpu-baseline --steps 3
# --warmup 3` (the mean of its 3 launches), ncu --metrics
# dram__bytes_read.sum,dram__bytes_write.sum --clock-control none.
# ---------------------------------------------------------------------------
NCU_TRAFFIC = {
    "find_kernel": {"bytes": 269957291, "sources": ("find.cu", "common.cuh", "launch.h"),
                    "sha256": "4dee867c0f4192e6"},
    "upsert_single_kernel": {"bytes": 330548651, "sources": ("upsert.cu", "common.cuh", "launch.h"),
                             "sha256": "df235f4f136a45f4"},
}


def ncu_traffic(kernel):
    import hashlib
    rec = NCU_TRAFFIC.get(kernel)
    if not rec or not rec["bytes"]:
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


def host_info():
    """The host's core count and CPU model (lscpu), for the CPU baseline."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class Ctx:
    """Device, stream, L2 flush buffer and helpers shared by the workloads."""

    def __init__(self, local):
        import torch

        import hash_table_cache_gb300 as hkv
        self.torch = torch
        self.hkv = hkv
        self.dev = torch.device("cuda", local)
        self.local = local
        self.stream = torch.cuda.current_stream()
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=self.dev)

    def dk(self, a):
        return self.torch.from_numpy(wl.as_i64(np.asarray(a, np.uint64))).to(self.dev)

    def ev(self):
        return self.torch.cuda.Event(enable_timing=True)

    def timed(self, fn):
        """One call between CUDA events on the current stream, L2 flushed
        before (outside the events)."""
        self.flush.zero_()
        a, b = self.ev(), self.ev()
        a.record(self.stream)
        fn()
        b.record(self.stream)
        b.synchronize()
        return a.elapsed_time(b) * 1e-3


def fill_table(ctx, t, target, pos, keys, dim, batch=FILL_BATCH):
    while t.size() < target and pos < keys.size:
        k = ctx.dk(keys[pos:pos + batch])
        t.insert_or_assign(k, wl.key_values_torch(k, dim, salt=1), None)
        pos += batch
    return pos


def resident_keys(t):
    return t.export(with_values=False)[0].cpu().numpy().view(np.uint64)


def c2_sweep(ctx, seed_base, peak):
    """find at each load factor on the filling table (80% hits drawn from the
    resident set), insert_or_assign at each load factor on re-filled tables
    (median of 3), each with its roofline fraction."""
    torch, hkv = ctx.torch, ctx.hkv
    keys = wl.unique_keys(3 + seed_base, 2 * CAP)
    sweep = {}
    t = hkv.HashTable(CAP, DIM, device=ctx.local)
    pos = 0
    vout = torch.empty((BATCH, DIM), dtype=torch.float32, device=ctx.dev)
    fout = torch.empty(BATCH, dtype=torch.uint8, device=ctx.dev)
    sout = torch.empty(BATCH, dtype=torch.int64, device=ctx.dev)
    for lam in LAMBDAS:
        pos = fill_table(ctx, t, lam * CAP, pos, keys, DIM)
        res = resident_keys(t)
        q, _ = wl.hit_mix(4 + seed_base, res, 5 + seed_base, BATCH, HIT)
        qd = ctx.dk(q)
        for _ in range(2):
            t.find(qd, vout, fout, sout)
        ft = [ctx.timed(lambda: t.find(qd, vout, fout, sout)) for _ in range(7)]
        f_med = statistics.median(ft)
        hit = float(fout.float().mean().item())
        fb = find_bytes_per_key(DIM, hit) * BATCH
        sweep[lam] = {"lambda_actual": t.size() / CAP, "find_bkvs": BATCH / f_med / 1e9,
                      "find_hit_rate": hit, "find_frac": fb / f_med / 1e9 / peak}
    t.close()
    for lam in LAMBDAS:
        ut, fr = [], []
        for rep in range(3):
            t = hkv.HashTable(CAP, DIM, device=ctx.local)
            fill_table(ctx, t, lam * CAP, 0, keys, DIM)
            # counts read before the batch is prepared: a synchronising call
            # right before a single timed call slows that call down
            c0 = t.op_counts()
            res = resident_keys(t)
            q, _ = wl.hit_mix(6 + seed_base + rep, res, 7 + seed_base + rep, BATCH, HIT)
            qd = ctx.dk(q)
            vd = wl.key_values_torch(qd, DIM, salt=2)
            dt = ctx.timed(lambda: t.insert_or_assign(qd, vd, None))
            c = {k: v - c0[k] for k, v in t.op_counts().items()}
            ut.append(dt)
            fr.append(upsert_bytes_paths(c, BATCH, DIM) / dt / 1e9 / peak)
            t.close()
        sweep[lam]["upsert_bkvs"] = BATCH / statistics.median(ut) / 1e9
        sweep[lam]["upsert_frac"] = statistics.median(fr)

    def variation(xs):
        return (max(xs) - min(xs)) / statistics.mean(xs)
    summary = {"find_bkvs_variation": variation([v["find_bkvs"] for v in sweep.values()]),
               "upsert_frac_variation": variation([v["upsert_frac"] for v in sweep.values()]),
               "definition": "(max - min) / mean over the load factors"}
    return sweep, summary


def c2_steps(ctx, args, seed_base, world):
    """The headline steps at load factor 1.0.  A twin table fed the same
    calls (single mode: identical contents) gives the resident set before and
    after each step's insert_or_assign, from which that step's hits are
    drawn, untimed."""
    torch, hkv = ctx.torch, ctx.hkv
    import torch.distributed as dist
    keys = wl.unique_keys(3 + seed_base, 2 * CAP)
    t = hkv.HashTable(CAP, DIM, device=ctx.local)
    twin = hkv.HashTable(CAP, DIM, device=ctx.local)
    fill_table(ctx, t, CAP, 0, keys, DIM)
    fill_table(ctx, twin, CAP, 0, keys, DIM)
    nsteps = args.warmup + args.steps
    up_k, up_v, fq = [], [], []
    res = resident_keys(twin)
    for s in range(nsteps):
        q, _ = wl.hit_mix(100 + s + seed_base, res, 200 + seed_base, BATCH, HIT,
                          fresh_start=s * BATCH)
        qd = ctx.dk(q)
        up_k.append(qd)
        up_v.append(wl.key_values_torch(qd, DIM, salt=3 + s))
        twin.insert_or_assign(up_k[s], up_v[s], None)
        res = resident_keys(twin)
        f, _ = wl.hit_mix(300 + s + seed_base, res, 400 + seed_base, BATCH, HIT,
                          fresh_start=s * BATCH)
        fq.append(ctx.dk(f))
    twin.close()
    vout = torch.empty((BATCH, DIM), dtype=torch.float32, device=ctx.dev)
    fout = torch.empty(BATCH, dtype=torch.uint8, device=ctx.dev)
    sout = torch.empty(BATCH, dtype=torch.int64, device=ctx.dev)
    ev = [[ctx.ev() for _ in range(3)] for _ in range(nsteps)]
    torch.cuda.synchronize()
    for s in range(args.warmup):
        ctx.flush.zero_()
        t.insert_or_assign(up_k[s], up_v[s], None)
        t.find(fq[s], vout, fout, sout)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t.reset_op_counts()
    hits = torch.zeros((), dtype=torch.float64, device=ctx.dev)
    with Clocks(ctx.local) as clk:
        w0 = time.time()
        # NVTX range "timed": lets a profiler select the timed launches
        torch.cuda.nvtx.range_push("timed")
        for s in range(args.warmup, nsteps):
            ctx.flush.zero_()
            e0, e1, e2 = ev[s]
            e0.record(ctx.stream)
            t.insert_or_assign(up_k[s], up_v[s], None)
            e1.record(ctx.stream)
            t.find(fq[s], vout, fout, sout)
            e2.record(ctx.stream)
            hits += fout.sum()  # outside the events
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        clk.mark(w0, time.time())
    if world > 1:
        dist.barrier()
    up_t = [ev[s][0].elapsed_time(ev[s][1]) * 1e-3 for s in range(args.warmup, nsteps)]
    fi_t = [ev[s][1].elapsed_time(ev[s][2]) * 1e-3 for s in range(args.warmup, nsteps)]
    counts = t.op_counts()
    hit_rate = float(hits.item()) / (BATCH * args.steps)
    return {"table": t, "up_k": up_k, "up_v": up_v, "fq": fq, "up_t": up_t, "fi_t": fi_t,
            "counts": counts, "hit_rate": hit_rate, "clocks": clk.summary(), "nsteps": nsteps}


def api_calls(ctx, st, peak):
    """The other calls of the API on the same full table, one 2^20-key batch
    each (median of 3, L2 flushed before each)."""
    torch, hkv = ctx.torch, ctx.hkv
    t, up_k, up_v, fq, nsteps = st["table"], st["up_k"], st["up_v"], st["fq"], st["nsteps"]
    api = {}
    qk, qv = fq[-1], up_v[-1]
    fout = torch.empty(BATCH, dtype=torch.uint8, device=ctx.dev)
    sout = torch.empty(BATCH, dtype=torch.int64, device=ctx.dev)
    ptr_out = torch.empty(BATCH, dtype=torch.int64, device=ctx.dev)
    api["contains_bkvs"] = BATCH / statistics.median(
        [ctx.timed(lambda: t.contains(qk)) for _ in range(3)]) / 1e9
    api["find_ptr_bkvs"] = BATCH / statistics.median(
        [ctx.timed(lambda: hkv.hkv_find_ptr(t.handle, BATCH, qk, ptr_out, fout, sout))
         for _ in range(3)]) / 1e9
    ta = statistics.median([ctx.timed(lambda: t.assign(qk, qv, None)) for _ in range(3)])
    api["assign_bkvs"] = BATCH / ta / 1e9
    # assign's algorithmic bytes: a hit as assign_bytes_per_hit, a miss its
    # key and digest line
    hits = int(t.contains(qk).sum().item())
    api["assign_frac"] = (hits * assign_bytes_per_hit(DIM)
                          + (BATCH - hits) * (8 + 128)) / ta / (peak * 1e9)
    ek = torch.empty(BATCH, dtype=torch.int64, device=ctx.dev)
    ev_ = torch.empty((BATCH, DIM), dtype=torch.float32, device=ctx.dev)
    es = torch.empty(BATCH, dtype=torch.int64, device=ctx.dev)
    ec = torch.zeros(1, dtype=torch.int64, device=ctx.dev)
    api["insert_and_evict_bkvs"] = BATCH / statistics.median(
        [ctx.timed(lambda: hkv.hkv_insert_and_evict(t.handle, BATCH, up_k[s], up_v[s], None, ek,
                                                     ev_, es, ec))
         for s in range(3)]) / 1e9
    fio_v = [qv.clone() for _ in range(3)]
    api["find_or_insert_bkvs"] = BATCH / statistics.median(
        [ctx.timed(lambda: t.find_or_insert(up_k[(s + 3) % nsteps], fio_v[s], None))
         for s in range(3)]) / 1e9
    return api


def end_to_end(ctx, st, ne, world):
    """End to end through the public API with host buffers: every step
    copies its inputs from pinned host memory, runs insert_or_assign + find
    and copies the find results back.  Copies run on their own streams,
    double buffered, so step s+1's upload and step s-1's download overlap
    step s.  Also times the same copies with no table work (the link alone,
    best of 3 runs: the link is shared with the machine's other work)."""
    torch = ctx.torch
    t, up_k, up_v, fq, nsteps = st["table"], st["up_k"], st["up_v"], st["fq"], st["nsteps"]
    stream = ctx.stream
    hk = [up_k[s % nsteps].cpu().pin_memory() for s in range(2)]
    hv = [up_v[s % nsteps].cpu().pin_memory() for s in range(2)]
    hq = [fq[s % nsteps].cpu().pin_memory() for s in range(2)]
    dk_ = [torch.empty_like(up_k[0]) for _ in range(2)]
    dv_ = [torch.empty_like(up_v[0]) for _ in range(2)]
    dq_ = [torch.empty_like(fq[0]) for _ in range(2)]
    ov_ = [torch.empty((BATCH, DIM), dtype=torch.float32, device=ctx.dev) for _ in range(2)]
    of_ = [torch.empty(BATCH, dtype=torch.uint8, device=ctx.dev) for _ in range(2)]
    os_ = [torch.empty(BATCH, dtype=torch.int64, device=ctx.dev) for _ in range(2)]
    hvo = [torch.empty((BATCH, DIM), dtype=torch.float32).pin_memory() for _ in range(2)]
    hfo = [torch.empty(BATCH, dtype=torch.uint8).pin_memory() for _ in range(2)]
    hso = [torch.empty(BATCH, dtype=torch.int64).pin_memory() for _ in range(2)]
    up_s, dn_s = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(ne)]
    done = [torch.cuda.Event() for _ in range(ne)]
    out_read = [torch.cuda.Event() for _ in range(ne)]
    torch.cuda.synchronize()
    a, b = ctx.ev(), ctx.ev()
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
    return {"value": 2 * BATCH * ne * world / e_total / 1e9, "unit": "B-KV/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "steps": ne, "overlap": "uploads and downloads on their own streams, double buffered",
            "link_only_s_per_step": link_total / ne,
            "frac_of_link_bound": link_total / e_total}


# ---------------------------------------------------------------------------
# The other workloads.  Each returns a dict with its throughput, per-call
# figures and roofline fractions (algorithmic bytes / time / measured peak).
# ---------------------------------------------------------------------------
OTHER = {
    "c1": "single-bucket, capacity 65,536, dim 8, one batch of 65,536 unique keys (score = index), "
          "then a find of 65,536 keys (half inserted)",
    "c3": "single-bucket, capacity 2^26, dim 64, load factor 1.0, steps of insert_or_assign 2^20 "
          "Zipf(1.05) over 2^32 keys (score = step) + find 2^20 from the same Zipf",
    "c4": "dual-bucket, capacity 2^26, dim 128, 1.5 x capacity unique keys with unique random "
          "scores inserted in 2^20 batches, then a find of 2^20 inserted keys",
    "c5": "tiered single-bucket, capacity 2^28, dim 64, 32 GiB of values in HBM and 32 GiB in mapped "
          "host memory, load factor 1.0; mixed stream on three CUDA streams: find 60%, assign 20%, "
          "insert_or_assign 20%, batches of 2^20, Zipf(1.1) over 2^34 keys",
}


def cfg_c1(ctx, steps, warmup, peak):
    torch, hkv = ctx.torch, ctx.hkv
    cap, dim, n = 65536, 8, 65536
    keys = wl.unique_keys(1, n)
    vals = wl.randn_values(0, n, dim, device=ctx.dev)
    sc = ctx.dk(np.arange(n, dtype=np.uint64))
    q = np.empty(n, np.uint64)
    q[0::2] = keys[0::2]
    q[1::2] = wl.unique_keys(2, n // 2)
    kd, qd = ctx.dk(keys), ctx.dk(q)
    up, fi, counts, hit = [], [], None, 0.0
    for s in range(warmup + steps):
        t = hkv.HashTable(cap, dim, device=ctx.local)
        ctx.flush.zero_()
        a, b, c = ctx.ev(), ctx.ev(), ctx.ev()
        a.record(ctx.stream)
        t.insert_or_assign(kd, vals, sc)
        b.record(ctx.stream)
        _, fo, _ = t.find(qd)
        c.record(ctx.stream)
        c.synchronize()
        if s >= warmup:
            up.append(a.elapsed_time(b) * 1e-3)
            fi.append(b.elapsed_time(c) * 1e-3)
            counts = t.op_counts()
            hit = float(fo.float().mean().item())
        t.close()
    u, f = statistics.mean(up), statistics.mean(fi)
    ub, fb = upsert_bytes_paths(counts, n, dim), find_bytes_per_key(dim, hit) * n
    return {"value": 2 * n / (u + f) / 1e9, "ms_per_step": (u + f) * 1e3,
            "insert_or_assign_bkvs": n / u / 1e9, "find_bkvs": n / f / 1e9,
            "insert_or_assign_frac": ub / u / 1e9 / peak, "find_frac": fb / f / 1e9 / peak,
            "find_hit_rate": hit, "op_counts": counts,
            "note": "the table fits in L2 (64 KiB digests, 1 MiB pairs, 2 MiB values): the "
                    "fractions measure the method's bytes, not DRAM traffic",
            "steps": steps, "gpu_launches_per_step": 4}


def cfg_c3(ctx, steps, warmup, peak, small=False):
    """small: 2^23 slots and 2^17-key batches (the same keys per bucket), a
    size a full profiler capture handles."""
    torch, hkv = ctx.torch, ctx.hkv
    cap, dim, n = (1 << 23, 64, 1 << 17) if small else (1 << 26, 64, 1 << 20)
    t = hkv.HashTable(cap, dim, device=ctx.local)
    keys = wl.unique_keys(6, int(1.6 * cap))
    fill_table(ctx, t, cap, 0, keys, dim, batch=1 << 20)
    del keys
    up, fi, ub, fb, uniq, hits = [], [], [], [], [], []
    fo = torch.empty(n, dtype=torch.uint8, device=ctx.dev)
    vo = torch.empty((n, dim), dtype=torch.float32, device=ctx.dev)
    so = torch.empty(n, dtype=torch.int64, device=ctx.dev)
    for s in range(warmup + steps):
        u = ctx.dk(wl.zipf_keys(7 + s, n, 1.05, 1 << 32))
        f = ctx.dk(wl.zipf_keys(10007 + s, n, 1.05, 1 << 32))
        c0 = t.op_counts()
        uv = wl.key_values_torch(u, dim, salt=100 + s)
        if s == warmup:
            torch.cuda.nvtx.range_push("timed")  # lets a profiler select the timed steps
        ctx.flush.zero_()
        a, b, c = ctx.ev(), ctx.ev(), ctx.ev()
        a.record(ctx.stream)
        t.insert_or_assign(u, uv, None)
        b.record(ctx.stream)
        t.find(f, vo, fo, so)
        c.record(ctx.stream)
        c.synchronize()
        if s >= warmup:
            du, df = a.elapsed_time(b) * 1e-3, b.elapsed_time(c) * 1e-3
            cnt = {k: v - c0[k] for k, v in t.op_counts().items()}
            h = float(fo.float().mean().item())
            up.append(du)
            fi.append(df)
            ub.append(upsert_bytes_paths(cnt, n, dim))
            fb.append(find_bytes_per_key(dim, h) * n)
            uniq.append(int(torch.unique(u).numel()))
            hits.append(h)
    torch.cuda.nvtx.range_pop()
    t.close()
    u, f = statistics.mean(up), statistics.mean(fi)
    return {"value": 2 * n / (u + f) / 1e9, "ms_per_step": (u + f) * 1e3,
            "insert_or_assign_bkvs": n / u / 1e9, "find_bkvs": n / f / 1e9,
            "insert_or_assign_frac": statistics.mean(ub) / u / 1e9 / peak,
            "find_frac": statistics.mean(fb) / f / 1e9 / peak,
            "unique_keys_per_batch": statistics.mean(uniq), "find_hit_rate": statistics.mean(hits),
            "steps": steps, "gpu_launches_per_step": 4}


def cfg_c4(ctx, steps, warmup, peak, small=False):
    """Dual mode: the 1.5 x capacity insert stream (every batch timed), the
    retention of the top-N scores after it, then finds of inserted keys.
    small: 2^23 slots and 2^17-key batches (the same keys per bucket); the
    batches at load factor 1.0 run inside an NVTX range "timed"."""
    torch, hkv = ctx.torch, ctx.hkv
    cap, dim, n = (1 << 23, 128, 1 << 17) if small else (1 << 26, 128, 1 << 20)
    nb = cap // 128
    t = hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_DUAL, device=ctx.local)
    total = int(1.5 * cap)
    keys = wl.unique_keys(8, total)
    scores = wl.stream(9, total) >> np.uint64(2)
    up_t, up_b, lam1 = [], [], []
    in_range = False
    for i, p in enumerate(range(0, total, n)):
        k = ctx.dk(keys[p:p + n])
        sc = ctx.dk(scores[p:p + n])
        v = wl.key_values_torch(k, dim, salt=1)
        c0 = t.op_counts()
        if not in_range and t.size() >= cap:
            torch.cuda.nvtx.range_push("timed")  # the batches at load factor 1.0
            in_range = True
        dt = ctx.timed(lambda: t.insert_or_assign(k, v, sc))
        cnt = {kk: vv - c0[kk] for kk, vv in t.op_counts().items()}
        up_t.append(dt)
        up_b.append(upsert_bytes_paths(cnt, k.numel(), dim, dual=True))
        lam1.append(cnt["evicted"] + cnt["rejected"] > 0)
    if in_range:
        torch.cuda.nvtx.range_pop()
    # top-N retention (HKV §5.5, Table 11): resident keys among the N = capacity
    # highest scores of all inserted keys (scores are distinct)
    thr = np.partition(scores, total - cap)[total - cap]
    rk, _, rs = t.export(with_values=False)
    retention = int((rs >= int(thr)).sum().item()) / cap  # scores < 2^62: no sign issue
    # absent keys with a candidate bucket that still has a free slot: Algorithm
    # 3 run key by key would have placed them (D1); counted on a sample
    ptrs, found, _ = t.find_ptr(rk, with_scores=False)
    info = t.info()
    occ = torch.bincount(rows_of_ptrs(ptrs, found, info) // 128, minlength=nb)
    smp = ctx.dk(keys[wl.permutation(11, total)[:1 << 20]])
    present = t.contains(smp).bool()
    absent = smp[~present]
    b1 = first_bucket_t(absent, nb)
    b2 = second_bucket_t(absent, b1, nb)
    d1_departures = int(((occ[b1] < 128) | (occ[b2] < 128)).sum().item())
    del rk, rs, ptrs, found
    # finds of inserted keys, hits split between first and second buckets
    fi, fb, hr = [], [], []
    for s in range(warmup + steps):
        q = ctx.dk(wl.choice(10 + s, keys, n))
        qp, qf, _ = t.find_ptr(q, with_scores=False)
        rows = rows_of_ptrs(qp, qf, info)
        first = qf.bool() & (rows // 128 == first_bucket_t(q, nb))
        n1 = int(first.sum().item())
        nh = int(qf.sum().item())
        vo = torch.empty((n, dim), dtype=torch.float32, device=ctx.dev)
        df = ctx.timed(lambda: t.find(q, vo, qf))
        if s >= warmup:
            fi.append(df)
            fb.append(find_bytes_dual(dim, n1, nh - n1, n - nh))
            hr.append(nh / n)
    t.close()
    l1 = [x for x, full in zip(up_t, lam1) if full]
    l1b = [x for x, full in zip(up_b, lam1) if full]
    f = statistics.mean(fi)
    return {"insert_or_assign_bkvs_all": total / sum(up_t) / 1e9,
            "insert_or_assign_bkvs_at_lambda_1": (len(l1) * n) / sum(l1) / 1e9 if l1 else None,
            "insert_or_assign_frac_at_lambda_1": (sum(l1b) / sum(l1) / 1e9 / peak) if l1 else None,
            "insert_batches": len(up_t), "batches_at_lambda_1": len(l1),
            "find_bkvs": n / f / 1e9, "find_frac": statistics.mean(fb) / f / 1e9 / peak,
            "find_hit_rate": statistics.mean(hr),
            "top_n_retention": retention,
            "absent_keys_sampled": int(absent.numel()),
            "absent_with_free_candidate": d1_departures,
            "value": (total + steps * n) / (sum(up_t) + sum(fi)) / 1e9,
            "steps": steps}


def cfg_c5(ctx, steps, warmup, peak, link, link_slab=None):
    """Tiered mixed stream: find, assign and insert_or_assign batches on
    three streams (3:1:1), ordered by the table's roles.  Link bound: the
    value bytes that cross the host link (rows of host-resident keys read by
    finds and written by assign / insert_or_assign) at the probed SM-access
    rates, against the HBM bytes at the copy peak.  `link`: random rows over
    a 1 GiB buffer (the link itself); `link_slab`: over a buffer the size of
    the table's 32 GiB slab, where the device's address translation of host
    memory, not the link, sets the rate of random rows."""
    torch, hkv = ctx.torch, ctx.hkv
    cap, dim, n = 1 << 28, 64, 1 << 20
    rb = 4 * dim
    t = hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_TIERED, value_hbm_bytes=32 << 30,
                      device=ctx.local)
    keys = wl.unique_keys(11, int(1.6 * cap))
    fill_table(ctx, t, cap, 0, keys, dim, batch=1 << 20)
    del keys
    info = t.info()
    host_share = 1 - info["hbm_value_rows"] / cap
    sf, sa, su = (torch.cuda.Stream() for _ in range(3))
    kinds = ["find", "find", "find", "assign", "upsert"]
    nsteps = warmup + steps
    plan = []
    for s in range(nsteps * 5):
        k = ctx.dk(wl.zipf_keys(12 + s, n, 1.1, 1 << 34))
        plan.append((kinds[s % 5], k, wl.key_values_torch(k, dim, salt=0)))
    outs = [(torch.empty((n, dim), device=ctx.dev), torch.empty(n, dtype=torch.uint8, device=ctx.dev))
            for _ in range(3)]
    torch.cuda.synchronize()
    times, host_rd, host_wr, hbm_b = [], [], [], []
    for s in range(nsteps):
        # untimed: the batches' hits in host rows (find* on the current table)
        rd = wr = fh = ah = 0
        for kind, k, _ in plan[5 * s:5 * s + 5]:
            p, fo, _ = t.find_ptr(k, with_scores=False)
            rows = rows_of_ptrs(p, fo, info)
            in_host = int((fo.bool() & (rows >= info["hbm_value_rows"])).sum().item())
            if kind == "find":
                rd += in_host
                fh += int(fo.sum().item())
            elif kind == "assign":
                wr += in_host
                ah += int(fo.sum().item())
        c0 = t.op_counts()
        a, b = ctx.ev(), ctx.ev()
        ctx.flush.zero_()
        a.record(ctx.stream)
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
            ctx.stream.wait_event(e)
        b.record(ctx.stream)
        b.synchronize()
        cnt = {kk: vv - c0[kk] for kk, vv in t.op_counts().items()}
        if s >= warmup:
            times.append(a.elapsed_time(b) * 1e-3)
            # insert_or_assign rows written to host memory: the host share of
            # the rows it wrote (its keys hash uniformly over the buckets);
            # the step's counts also hold the assign's updates
            up_rows = max(cnt["updated"] + cnt["admitted"] - ah, 0)
            host_rd.append(rd * rb)
            host_wr.append(wr * rb + host_share * up_rows * rb)
            hbm_b.append(find_bytes_per_key(dim, fh / (3 * n)) * 3 * n
                         + upsert_bytes_paths(cnt, 2 * n, dim) - (rd + wr) * rb)
    t.close()
    step = statistics.mean(times)
    rd_b, wr_b, hb = statistics.mean(host_rd), statistics.mean(host_wr), statistics.mean(hbm_b)
    link_s = (rd_b / link["row_read"] + wr_b / link["row_write"]) if link.get("row_read") else None
    hbm_s = hb / (peak * 1e9)
    bound = max(x for x in (link_s, hbm_s) if x is not None)
    out = {"value": 5 * n / step / 1e9, "ms_per_step": step * 1e3,
           "host_read_bytes_per_step": rd_b, "host_write_bytes_per_step": wr_b,
           "hbm_bytes_per_step": hb, "link_bound_s": link_s, "hbm_bound_s": hbm_s,
           "frac_of_bound": bound / step,
           "bound": "host link" if link_s and link_s >= hbm_s else "hbm",
           "link": "SM loads/stores over pinned host memory (a host-NUMA memory pool; "
                   "NVLink-C2C on a Grace host)",
           "steps": steps, "gpu_launches_per_step": 9}
    if link_slab and link_slab.get("row_read") and link_slab.get("row_write"):
        slab_s = rd_b / link_slab["row_read"] + wr_b / link_slab["row_write"]
        # uniform random rows over a slab this size: the skewed stream's hot
        # rows stay in L2, so this is context for the slab's memory, not a
        # bound on the step
        out["slab_uniform_row_rates_bytes_per_s"] = link_slab
        out["slab_uniform_rows_s"] = slab_s
    return out


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    ctx = Ctx(local)
    ctx.hkv.load()
    seed_base = replica_seed_base(rank)
    peak, peak_kind = read_peaks()

    sweep, sweep_summary = ({}, None) if args.skip_sweep else c2_sweep(ctx, seed_base, peak)
    st = c2_steps(ctx, args, seed_base, world)
    up_t, fi_t, counts = st["up_t"], st["fi_t"], st["counts"]
    total = sum(up_t) + sum(fi_t)
    total, value = job_time_and_value(total, 2 * BATCH * args.steps, world, dev)

    # roofline: find is one kernel per call, timed exactly by the events
    # around hkv_find; insert_or_assign is a call of three kernels (clear,
    # stage, bucket pass) and is reported as a call
    hit_rate = st["hit_rate"]
    f_avg, u_avg = statistics.mean(fi_t), statistics.mean(up_t)
    fb = find_bytes_per_key(DIM, hit_rate) * BATCH
    per_call = {k: v / args.steps for k, v in counts.items()}
    rows = per_call["updated"] + per_call["admitted"]
    ub = upsert_bytes(BATCH, DIM, CAP // 128, rows, False)
    ub_paths = upsert_bytes_paths(per_call, BATCH, DIM)
    find_roof = {"bound": "hbm", "achieved": fb / f_avg / 1e9, "peak": peak, "unit": "GB/s",
                 "frac": fb / f_avg / 1e9 / peak, "traffic": ncu_traffic("find_kernel"),
                 "kernel": "find_kernel",
                 "bytes_per_launch": fb, "avg_launch_s": f_avg, "peak_kind": peak_kind}
    up_traffic = ncu_traffic("upsert_single_kernel")
    up_roof = {"bound": "hbm", "achieved": ub / u_avg / 1e9, "peak": peak, "unit": "GB/s",
               "frac": ub / u_avg / 1e9 / peak,
               "frac_survey_model": ub_paths / u_avg / 1e9 / peak,
               "bytes_survey_model": ub_paths,
               "traffic": None if up_traffic is None else {"upsert_single_kernel": up_traffic},
               "kernel": "insert_or_assign call (clear + stage_kernel + upsert_single_kernel)",
               "bytes_per_launch": ub, "avg_launch_s": u_avg, "peak_kind": peak_kind,
               "models": "frac: this build's slot layout (per touched bucket 2 KiB of pairs + "
                         "2 x 128 B digest line, per changed slot 16 B + a row); "
                         "frac_survey_model: per-path algorithmic bytes from the call's outcome "
                         "counts"}
    try:
        rates = probe_access_rates((32, 128, 4 * DIM))
        rcounts = find_random_counts(BATCH, DIM, hit_rate, CAP // 128)
        seq = BATCH * (8 + hit_rate * (4 * DIM + 8) + 1)
        ff = access_floor(rcounts, seq, rates, peak)
        access = {"random_reads_per_s": {f"{g}B": v["plateau"] for g, v in rates.items()},
                  "probe_grid": {f"{g}B": v["grid"] for g, v in rates.items()},
                  "find": {"floor_s": ff, "measured_s": f_avg, "frac": ff / f_avg},
                  "note": "floor = random accesses at the probed plateau rates (best over reads "
                          "in flight and blocks per SM) + streamed bytes at the copy peak"}
    except Exception as exc:  # the probe is a measurement aid; the line stands without it
        access = {"unavailable": str(exc)}
    api = api_calls(ctx, st, peak)
    e2e = end_to_end(ctx, st, args.steps, world) if (rank == 0 or world > 1) else None
    st["table"].close()
    clocks = st["clocks"]

    configs = {}
    if not args.skip_configs and rank == 0:
        link = {}
        try:
            link = probe_host_link(4 * 64)
            link_slab = probe_host_link(4 * 64, 32 << 30, kinds=slab_kinds(32 << 30))
        except Exception as exc:
            link, link_slab = {"unavailable": str(exc)}, {}
        configs["host_link_bytes_per_s"] = link
        configs["host_link_bytes_per_s_32GiB"] = link_slab
        for name, fn in (("c1", lambda: cfg_c1(ctx, 5, 3, peak)),
                         ("c3", lambda: cfg_c3(ctx, args.config_steps, 3, peak)),
                         ("c4", lambda: cfg_c4(ctx, args.config_steps, 3, peak)),
                         ("c5", lambda: cfg_c5(ctx, min(args.config_steps, 3), 2, peak, link,
                                              link_slab))):
            try:
                configs[name] = {"workload": OTHER[name], **fn()}
            except Exception as exc:
                configs[name] = {"workload": OTHER[name], "unavailable": f"{type(exc).__name__}: {exc}"}
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds, with_dual=not args.skip_configs)
        if "c4" in configs and cpu.get("dual_retention_scaled"):
            configs["c4"]["retention_scaled"] = cpu["dual_retention_scaled"]
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
                   "hits_drawn_from": "the resident set before (insert) and after (find) each "
                                      "step's insert_or_assign",
                   "l2": "flushed between steps (256 MiB write), flush outside timed events",
                   "parallelism": f"replicas x{world}"},
        "roofline": find_roof,
        "roofline_all": {"find": find_roof, "insert_or_assign": up_roof},
        "access_ceiling": access,
        "per_step": {"insert_or_assign_s": u_avg, "find_s": f_avg,
                     "find_bkvs": BATCH / f_avg / 1e9, "upsert_bkvs": BATCH / u_avg / 1e9,
                     "find_hit_rate": hit_rate, "op_counts": counts},
        "lambda_sweep": {str(k): v for k, v in sweep.items()},
        "lambda_sweep_summary": sweep_summary,
        "api_at_load_factor_1": api,
        "configs": configs,
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        # clear_scratch_kernel + stage_kernel + upsert_single_kernel + find_kernel
        "gpu_launches": args.steps * 4,
    }
    print(json.dumps(line))


def run_other(args):
    """One measurement line for one of the other workloads."""
    import torch
    torch.cuda.set_device(0)
    ctx = Ctx(0)
    ctx.hkv.load()
    peak, _ = read_peaks()
    cfg = args.config
    if cfg == "c1":
        r = cfg_c1(ctx, args.steps, args.warmup, peak)
    elif cfg == "c3":
        r = cfg_c3(ctx, args.steps, args.warmup, peak, small=args.small)
    elif cfg == "c4":
        r = cfg_c4(ctx, args.steps, args.warmup, peak, small=args.small)
    else:
        r = cfg_c5(ctx, args.steps, args.warmup, peak, probe_host_link(4 * 64),
                   probe_host_link(4 * 64, 32 << 30, kinds=slab_kinds(32 << 30)))
    line = {
        "metric": METRIC, "value": r["value"], "unit": "B-KV/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r.get("ms_per_step"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u64 keys/scores, f32 values (copied)", "data": "synthetic",
        "config": {"workload": OTHER[cfg], "name": cfg,
                   "scale": "2^23 slots, 2^17-key batches" if args.small and cfg in ("c3", "c4")
                   else "full",
                   "l2": "flushed before each timed call or step, outside the events"},
        "result": r,
    }
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


def dual_retention_scaled():
    """The dual-bucket stream scaled to 2^20 slots (8,192 buckets), dim 8: 1.5
    x capacity unique keys with unique random scores in 2^16 batches, on the
    oracle (Algorithm 3 key by key) and on the GPU; each side's share of the
    N = capacity highest scores that stays resident (HKV §5.5, Table 11)."""
    import torch

    import hash_table_cache_gb300 as hkv
    import oracle
    cap, dim, bs = 1 << 20, 8, 1 << 16
    total = int(1.5 * cap)
    keys = wl.unique_keys(8, total)
    scores = wl.stream(9, total) >> np.uint64(2)
    top = set(keys[np.argsort(scores)[-cap:]].tolist())
    o = oracle.OracleTable(cap // 128, dim, dual=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    t = hkv.HashTable(cap, dim, mode=hkv.HKV_MODE_DUAL, device=dev.index)
    t0 = time.perf_counter()
    for p in range(0, total, bs):
        k, s = keys[p:p + bs], scores[p:p + bs]
        v = wl.key_values(k, dim, salt=1)
        o.insert_or_assign(k, v, s)
    o_s = time.perf_counter() - t0
    for p in range(0, total, bs):
        k = torch.from_numpy(wl.as_i64(keys[p:p + bs])).to(dev)
        s = torch.from_numpy(wl.as_i64(scores[p:p + bs])).to(dev)
        t.insert_or_assign(k, wl.key_values_torch(k, dim, salt=1), s)
    gk = t.export(with_values=False)[0].cpu().numpy().view(np.uint64)
    t.close()
    ok = o.export()[0]
    return {"capacity": cap, "gpu": len(top & set(gk.tolist())) / cap,
            "oracle": len(top & set(ok.tolist())) / cap, "oracle_s": o_s}


def cpu_baseline(seconds, with_dual=False):
    rate, n, _, nk = oracle_step_rate(seconds)
    hi = host_info()
    out = {"value": rate / 1e9, "unit": "B-KV/s", "cores": 1, "kind": "oracle",
           "host": hi,
           "sample": f"{n} step(s) of insert_or_assign + find restricted to every "
                     f"{SAMPLE_EVERY}th bucket of the 2^22-slot table at load factor 1.0 "
                     f"(~{int(statistics.mean(nk))} keys per step; fill untimed), single-threaded "
                     f"on 1 of {hi['nproc']} host cores ({hi['cpu_model']})"}
    if with_dual:
        try:
            out["dual_retention_scaled"] = dual_retention_scaled()
        except Exception as exc:
            out["dual_retention_scaled"] = {"unavailable": str(exc)}
    return out


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    rate, n, times, nk = oracle_step_rate(None, steps=args.warmup + args.steps)
    w = args.warmup if len(times) > args.warmup else 0
    timed, tk = times[w:], nk[w:]
    value = sum(tk) / sum(timed) / 1e9
    hi = host_info()
    line = {
        "metric": METRIC, "value": value, "unit": "B-KV/s", "n_gpus": world, "steps": len(timed),
        "warmup": args.warmup, "ms_per_step": sum(timed) / len(timed) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u64 keys/scores, f32 values (copied)", "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD, "capacity": CAP, "dim": DIM, "batch": BATCH,
                   "hit_rate": HIT, "load_factor": 1.0, "mode": "single",
                   "parallelism": "cpu, 1 thread"},
        "cpu_baseline": {"value": value, "unit": "B-KV/s", "cores": 1, "kind": "oracle", "host": hi,
                         "sample": f"{len(timed)} timed step(s) of insert_or_assign + find "
                                   f"restricted to every {SAMPLE_EVERY}th bucket of the 2^22-slot "
                                   f"table at load factor 1.0 (~{int(statistics.mean(tk))} "
                                   f"keys/step), single-threaded on 1 of {hi['nproc']} host cores"},
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
    ctx = Ctx(0)
    keys = wl.unique_keys(3, 2 * CAP)
    t = hkv.HashTable(CAP, DIM)
    pos, out = 0, {}
    vout = torch.empty((BATCH, DIM), dtype=torch.float32, device=ctx.dev)
    fo = torch.empty(BATCH, dtype=torch.uint8, device=ctx.dev)
    so = torch.empty(BATCH, dtype=torch.int64, device=ctx.dev)
    for lam in ((0.5, 1.0) if what == "find" else (1.0,)):
        pos = fill_table(ctx, t, lam * CAP, pos, keys, DIM)
        res = resident_keys(t)
        if what == "find":
            for hit in (0.0, 0.8, 1.0):
                q, _ = wl.hit_mix(4, res, 5, BATCH, hit, fresh_start=(1 + int(lam * 4)) << 24)
                qd = ctx.dk(q)
                for _ in range(3):
                    t.find(qd, vout, fo, so)
                ts = [ctx.timed(lambda: t.find(qd, vout, fo, so)) for _ in range(5)]
                out[f"find lambda={lam} hits={hit}"] = BATCH / statistics.median(ts) / 1e9
        else:
            batches, prev = [], res
            for r in range(13):
                q, _ = wl.hit_mix(100 + r, prev, 200, BATCH, HIT, fresh_start=r * BATCH)
                prev = q
                qd = ctx.dk(q)
                batches.append((qd, wl.key_values_torch(qd, DIM, salt=3 + r)))
            torch.cuda.synchronize()
            ts = [ctx.timed(lambda: t.insert_or_assign(k, v, None)) for k, v in batches]
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


def run_probe_sweep():
    """Random reads of 32..512-byte granules over a 4 GiB buffer at 1..16
    reads in flight and 2, 4, 8 blocks per SM (G reads/s), the host link by
    SM loads and stores (GB/s), and random host rows by buffer size and
    memory kind (GB/s)."""
    import ctypes

    import torch
    torch.cuda.init()
    lib = _probe_lib()
    grid = {}
    for g in (32, 64, 128, 256, 512):
        for b in (2, 4, 8):
            for d in (1, 2, 4, 8, 16):
                if g >= 256 and d == 16:
                    continue  # 64 registers of rows per lane
                r = ctypes.c_double(0.0)
                st = lib.hkv_probe_random_reads_at(g, 4 << 30, d, b, ctypes.byref(r))
                grid[f"{g}B blocks={b} depth={d}"] = round(r.value / 1e9, 2) if st == 0 else None
    link = {k: (round(v / 1e9, 1) if v else None) for k, v in probe_host_link(256).items()}
    # random 256-byte rows over host buffers of growing size, mapped memory
    # and host-NUMA pool memory (the two kinds a tiered slab can be)
    slab = {}
    for gib in (1, 8, 16, 17, 18, 20, 24, 32):
        for kinds, name in (((2, 3), "mapped"), ((6, 7), "pool")):
            if name == "pool" and gib not in (1, 8, 16, 32):
                continue
            r = probe_host_link(256, gib << 30, kinds=kinds)
            slab[f"{name} {gib} GiB"] = {k: (round(v / 1e9, 1) if v else None) for k, v in r.items()}
    print(json.dumps({"random_reads_G_per_s": grid, "host_link_GB_per_s": link,
                      "host_rows_by_buffer_size_GB_per_s": slab}))


POLICY_SWEEP_ALPHAS = (0.5, 0.75, 0.99, 1.25)


def run_policy_sweep(args):
    """Cache hit rate by score policy and Zipf exponent (HKV §5.4 Exp #3c,
    Table 8): a 2^27-slot single-bucket table of 32-float rows (the pages'
    Config B), keys Zipf(alpha) over 2^32, batches of 2^20.  The table is
    warmed up with 2 x capacity keys of the stream (it fills to load factor
    1.0 and turns over once), then each of `args.steps` batches is looked up
    (contains: a hit is a key found) and inserted (insert_or_assign with the
    policy's score: customized gets the step as its score, the epoch
    policies a new epoch every step).  Also each policy's rate over the
    measured steps (lookups + inserts per second).  One JSON object."""
    import torch
    ctx = Ctx(0)
    hkv = ctx.hkv
    hkv.load()
    cap, dim, n, universe, warm_batch = 1 << 27, 32, 1 << 20, 1 << 32, 1 << 23
    policies = (("customized", hkv.HKV_POLICY_CUSTOMIZED), ("lru", hkv.HKV_POLICY_LRU),
                ("lfu", hkv.HKV_POLICY_LFU), ("epoch_lru", hkv.HKV_POLICY_EPOCH_LRU),
                ("epoch_lfu", hkv.HKV_POLICY_EPOCH_LFU))
    zeros = torch.zeros((warm_batch, dim), device=ctx.dev)  # values do not affect hits
    hit_rate = {name: {} for name, _ in policies}
    rate = {name: [] for name, _ in policies}
    for ai, alpha in enumerate(POLICY_SWEEP_ALPHAS):
        warm = [wl.zipf_keys_torch(1000 + 100 * ai + i, warm_batch, alpha, universe, ctx.dev)
                for i in range(2 * cap // warm_batch)]
        meas = [wl.zipf_keys_torch(2000 + 100 * ai + i, n, alpha, universe, ctx.dev)
                for i in range(args.steps)]
        for name, code in policies:
            t = hkv.HashTable(cap, dim, mode=code, device=ctx.local)
            step = 0

            def put(k):
                nonlocal step
                step += 1
                if name.startswith("epoch"):
                    t.set_epoch(step)
                sc = (torch.full((k.numel(),), step, dtype=torch.int64, device=ctx.dev)
                      if name == "customized" else None)
                t.insert_or_assign(k, zeros[:k.numel()], sc)

            for k in warm:
                put(k)
            hits = torch.zeros((), dtype=torch.int64, device=ctx.dev)
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            for k in meas:
                hits += t.contains(k).sum()
                put(k)
            b.record()
            b.synchronize()
            hit_rate[name][str(alpha)] = round(float(hits.item()) / (args.steps * n), 4)
            rate[name].append(2 * n * args.steps / (a.elapsed_time(b) * 1e-3) / 1e9)
            t.close()
        del warm, meas
    print(json.dumps({
        "workload": "single-bucket, capacity 2^27, dim 32 (Config B); Zipf(alpha) over 2^32 in "
                    "batches of 2^20; warm-up 2 x capacity stream keys, then "
                    f"{args.steps} batches each looked up (contains) and inserted",
        "hit_rate": hit_rate,
        "lookups_and_inserts_bkvs": {k: round(statistics.median(v), 3) for k, v in rate.items()},
        "data": "synthetic"}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--skip-sweep", action="store_true", help="no load-factor sweep")
    ap.add_argument("--skip-configs", action="store_true",
                    help="no other workloads (c1, c3, c4, c5) in the headline line")
    ap.add_argument("--config-steps", type=int, default=5,
                    help="timed steps of each other workload in the headline line")
    ap.add_argument("--config", default="c2", choices=["c1", "c2", "c3", "c4", "c5"],
                    help="workload; c2 (the default) is the headline line")
    ap.add_argument("--small", action="store_true",
                    help="c3, c4: 2^23 slots and 2^17-key batches (the same keys per bucket; "
                         "for profiler captures)")
    ap.add_argument("--probe-sweep", action="store_true",
                    help="print the random-read rates of this GPU over granule, reads in flight "
                         "and blocks per SM, and the host link by SM access, as one JSON object")
    ap.add_argument("--policy-sweep", action="store_true",
                    help="cache hit rate by score policy and Zipf exponent on a 2^27-slot table "
                         "(the pages' Table 8), as one JSON object; --steps measured batches")
    ap.add_argument("--ablation", choices=["digest", "pipeline"],
                    help="compare the default build with a variant build instead: find without "
                         "the digest line, or the pipelined bucket kernel")
    ap.add_argument("--ablation-child", help=argparse.SUPPRESS)
    ap.add_argument("--ablation-what", default="find", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.probe_sweep:
        run_probe_sweep()
    elif args.policy_sweep:
        run_policy_sweep(args)
    elif args.ablation_child:
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
