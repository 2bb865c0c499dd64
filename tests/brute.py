"""Brute-force models used to pin the oracle on tiny inputs (pure Python).

These are written independently of ``oracle/hkv_oracle.cpp`` and in a
different form:

* single-bucket mode uses the closed form of HierarchicalKV §3.3 (Algorithm 2)
  under the batch reading "resident keys update first, then absent keys":
  after a call, bucket b holds the 128 highest-ranked of (its residents after
  the in-place updates) plus (the absent keys hashed to it); rank = (score,
  key is new to the table in this call, key) -- an incoming key beats an
  older entry of equal score, as Algorithm 2 admits on score >= minimum.
  No slot, no arg-min loop, no eviction step.
* dual-bucket mode replays HierarchicalKV §3.4 (Algorithm 3) key by key on
  Python dicts.
* score policies (kLru, kLfu, kEpochLru, kEpochLfu, kCustomized; HKV §3.3 and
  Table 8 name them, the update rules are the oracle's reading R10) are
  computed with Python integers, saturation as a plain ``min``.
"""
from __future__ import annotations

import numpy as np

MASK = (1 << 64) - 1
RESERVED_LO = 0xFFFFFFFFFFFFFFF0
SLOTS = 128
CUSTOMIZED, LRU, LFU, EPOCH_LRU, EPOCH_LFU = range(5)
LOW32 = (1 << 32) - 1


def fmix64(h: int) -> int:
    h &= MASK
    h ^= h >> 33
    h = (h * 0xFF51AFD7ED558CCD) & MASK
    h ^= h >> 33
    h = (h * 0xC4CEB9FE1A85EC53) & MASK
    h ^= h >> 33
    return h


class BruteTable:
    def __init__(self, num_buckets: int, dim: int, dual: bool = False, policy: int = CUSTOMIZED):
        self.B = num_buckets
        self.dim = dim
        self.dual = dual
        self.policy = policy
        self.epoch = 0
        self.step = 1
        # bucket -> {key: (score, tuple(values))}
        self.bk = {b: {} for b in range(num_buckets)}

    # -- placement -------------------------------------------------------
    def b1(self, k):
        return fmix64(k) % self.B

    def b2(self, k):
        b1 = self.b1(k)
        b2 = fmix64(k ^ 0x9E3779B97F4A7C15) % self.B
        return (b1 + 1) % self.B if b2 == b1 else b2

    def where(self, k):
        if k in self.bk[self.b1(k)]:
            return self.b1(k)
        if self.dual and k in self.bk[self.b2(k)]:
            return self.b2(k)
        return None

    # -- helpers -----------------------------------------------------------
    @staticmethod
    def _last(keys):
        last, reserved = {}, 0
        for i, k in enumerate(keys):
            k = int(k)
            if k >= RESERVED_LO:
                reserved += 1
                continue
            last[k] = i
        return sorted(last.values()), reserved

    def residents(self):
        return {k for b in self.bk.values() for k in b}

    def _rule(self, keys, scores):
        """score(i, key, old score or None) for one call that writes scores."""
        pol, clock, hi = self.policy, self.step, self.epoch << 32
        if pol in (LRU, EPOCH_LRU) or (pol == CUSTOMIZED and scores is None):
            self.step += 1
        total = {}
        if pol in (LFU, EPOCH_LFU):
            for i, k in enumerate(keys):
                if k < RESERVED_LO:
                    total[k] = total.get(k, 0) + (int(scores[i]) if scores is not None else 1)

        def score(i, k, old):
            if pol == LRU:
                return clock
            if pol == EPOCH_LRU:
                return hi + clock % (1 << 32)
            if pol == LFU:
                return min((0 if old is None else old) + total[k], MASK)
            if pol == EPOCH_LFU:
                return hi + min((0 if old is None else old % (1 << 32)) + total[k], LOW32)
            return int(scores[i]) if scores is not None else clock
        return score

    # -- operations --------------------------------------------------------
    def insert_or_assign(self, keys, values, scores=None, update_resident=True, evicted_out=None):
        """update_resident=False: find_or_insert's insertion step (resident
        keys untouched).  evicted_out: list receiving (key, score, values) of
        the entries resident before the call and displaced by it."""
        keys = [int(k) for k in keys]
        values = np.asarray(values, np.float32).reshape(len(keys), self.dim)
        order, reserved = self._last(keys)
        score = self._rule(keys, scores)
        before = self.residents()
        updated = 0
        absent = []
        for i in order:
            k = keys[i]
            b = self.where(k)
            if b is not None:
                if update_resident:
                    self.bk[b][k] = (score(i, k, self.bk[b][k][0]), tuple(values[i].tolist()))
                    updated += 1
            else:
                absent.append(i)
        snapshot = {k: sv for d in self.bk.values() for k, sv in d.items()}
        if self.dual:
            for i in absent:
                self._dual_insert(keys[i], score(i, keys[i], None), tuple(values[i].tolist()))
        else:
            new = {keys[i] for i in absent}
            for i in absent:
                k = keys[i]
                self.bk[self.b1(k)][k] = (score(i, k, None), tuple(values[i].tolist()))
            for b, d in self.bk.items():
                if len(d) > SLOTS:
                    top = sorted(d.items(), key=lambda kv: (kv[1][0], kv[0] in new, kv[0]),
                                 reverse=True)[:SLOTS]
                    self.bk[b] = dict(top)
        after = self.residents()
        if evicted_out is not None:
            evicted_out.extend((k, snapshot[k][0], snapshot[k][1]) for k in sorted(before - after))
        absent_keys = {keys[i] for i in absent}
        return {
            "updated": updated,
            "admitted": len(absent_keys & after),
            "rejected": len(absent_keys - after),
            "evicted": len(before - after),
            "reserved": reserved,
        }

    def _dual_insert(self, k, s, v):
        x, y = self.b1(k), self.b2(k)
        dx, dy = self.bk[x], self.bk[y]
        if len(dx) < SLOTS or len(dy) < SLOTS:
            (dy if len(dy) < len(dx) else dx)[k] = (s, v)
            return
        mx = min(dx.items(), key=lambda kv: (kv[1][0], kv[0]))
        my = min(dy.items(), key=lambda kv: (kv[1][0], kv[0]))
        rx, ry = (mx[1][0], mx[0]), (my[1][0], my[0])
        d, m, r = (dy, my, ry) if ry < rx else (dx, mx, rx)
        if (s, k) > r:
            del d[m[0]]
            d[k] = (s, v)

    def assign(self, keys, values, scores=None):
        keys = [int(k) for k in keys]
        values = np.asarray(values, np.float32).reshape(len(keys), self.dim)
        order, _ = self._last(keys)
        keep = self.policy == CUSTOMIZED and scores is None
        score = None if keep else self._rule(keys, scores)
        for i in order:
            b = self.where(keys[i])
            if b is None:
                continue
            old = self.bk[b][keys[i]]
            s = old[0] if keep else score(i, keys[i], old[0])
            self.bk[b][keys[i]] = (s, tuple(values[i].tolist()))

    def erase(self, keys):
        for k in keys:
            k = int(k)
            if k >= RESERVED_LO:
                continue
            b = self.where(k)
            if b is not None:
                del self.bk[b][k]

    def find_or_insert(self, keys, values, scores=None):
        c = self.insert_or_assign(keys, values, scores, update_resident=False)
        vals = np.asarray(values, np.float32).reshape(len(keys), self.dim).copy()
        fv, found, _ = self.find(keys)
        vals[found.astype(bool)] = fv[found.astype(bool)]
        return c, vals, found

    def find(self, keys):
        n = len(keys)
        vals = np.zeros((n, self.dim), np.float32)
        found = np.zeros(n, np.uint8)
        scs = np.zeros(n, np.uint64)
        for i, k in enumerate(keys):
            k = int(k)
            if k >= RESERVED_LO:
                continue
            b = self.where(k)
            if b is None:
                continue
            s, v = self.bk[b][k]
            vals[i] = v
            found[i] = 1
            scs[i] = s
        return vals, found, scs

    def export(self):
        items = sorted((k, s, v) for d in self.bk.values() for k, (s, v) in d.items())
        keys = np.array([t[0] for t in items], np.uint64)
        scs = np.array([t[1] for t in items], np.uint64)
        vals = np.array([t[2] for t in items], np.float32).reshape(len(items), self.dim)
        return keys, vals, scs

    def size(self):
        return sum(len(d) for d in self.bk.values())
