"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module generates keys, scores and values only.  It holds none of the
table's own arithmetic (no bucket hash, no digest, no rank rule), so the CUDA
library and the CPU oracle can both be fed from it without sharing code.

Generators (all deterministic functions of their seed):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) for every 64-bit stream.  Its output function is a
  bijection of the 64-bit state and the state walks a full 2^64 cycle, so the
  first 2^64 outputs of one stream are pairwise distinct: that is how
  ``unique_keys`` gets distinct keys without a set.
* Zipf ranks by rejection-inversion (Hörmann and Derflinger, "Rejection-
  inversion to generate variates from monotone discrete distributions", ACM
  TOMACS 1996), vectorised over numpy.
* N(0,1) value rows from a seeded ``torch.Generator`` (``randn_values``), or
  rows that are a pure function of the key (``key_values``), so that a table
  row can be checked against its key anywhere without keeping the batch.

Keys never fall in the table's 16 reserved sentinel values
(0xFFFFFFFFFFFFFFF0 and above); a generator that would emit one raises.
"""
from __future__ import annotations

import numpy as np

GAMMA = 0x9E3779B97F4A7C15          # SplitMix64 state increment
_M1 = 0xBF58476D1CE4E5B9             # SplitMix64 output-mix multipliers
_M2 = 0x94D049BB133111EB
RESERVED_LO = 0xFFFFFFFFFFFFFFF0

_U = np.uint64


def mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (a bijection on uint64), elementwise."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> _U(30))) * _U(_M1)
        z = (z ^ (z >> _U(27))) * _U(_M2)
        return z ^ (z >> _U(31))


def _state0(seed: int) -> np.uint64:
    # Spread small integer seeds over the 2^64 cycle so that streams of
    # different seeds start far apart.
    return mix(np.array([int(seed) & 0xFFFFFFFFFFFFFFFF], np.uint64))[0]


def stream(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+n-1 of the SplitMix64 stream for ``seed``."""
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = _state0(seed) + idx * _U(GAMMA)
    return mix(state)


def _check_keys(keys: np.ndarray) -> np.ndarray:
    if keys.size and int(keys.max()) >= RESERVED_LO:
        raise RuntimeError("generator produced a reserved sentinel key; choose another seed")
    return keys


def unique_keys(seed: int, n: int, start: int = 0) -> np.ndarray:
    """n distinct uniform uint64 keys: positions start.. of the seed's stream."""
    return _check_keys(stream(seed, n, start))


def uniform01(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Doubles in [0, 1) from the top 53 bits of the stream."""
    return (stream(seed, n, start) >> _U(11)).astype(np.float64) * (1.0 / (1 << 53))


def permutation(seed: int, n: int) -> np.ndarray:
    """A seeded permutation of 0..n-1 (argsort of n stream values)."""
    return np.argsort(stream(seed, n), kind="stable")


def choice(seed: int, pool: np.ndarray, n: int) -> np.ndarray:
    """n uniform draws, with replacement, from ``pool``."""
    pool = np.asarray(pool)
    if pool.size == 0:
        raise ValueError("empty pool")
    idx = stream(seed, n) % _U(pool.size)
    return pool[idx.astype(np.int64)]


def hit_mix(seed: int, resident: np.ndarray, fresh_seed: int, n: int, hit_rate: float,
            fresh_start: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """A batch of n keys: round(hit_rate*n) drawn uniformly from ``resident``,
    the rest fresh (unique stream of ``fresh_seed``), then shuffled.
    Returns (keys, is_drawn_from_resident)."""
    n_hit = int(round(hit_rate * n))
    hits = choice(seed, resident, n_hit).astype(np.uint64)
    fresh = unique_keys(fresh_seed, n - n_hit, fresh_start)
    keys = np.concatenate([hits, fresh])
    drawn = np.concatenate([np.ones(n_hit, bool), np.zeros(n - n_hit, bool)])
    p = permutation(seed ^ 0x5DEECE66D, n)
    return keys[p], drawn[p]


# --------------------------------------------------------------------------
# Zipf by rejection-inversion.
# --------------------------------------------------------------------------
class Zipf:
    """Zipf(alpha) over ranks 1..universe, P(r) proportional to r^-alpha."""

    def __init__(self, alpha: float, universe: int):
        if alpha <= 0 or alpha == 1.0:
            raise ValueError("alpha must be > 0 and != 1")
        self.q = float(alpha)
        self.n = int(universe)
        self.hx1 = self._H(1.5) - 1.0
        self.hn = self._H(self.n + 0.5)
        self.s = 2.0 - self._Hinv(self._H(2.5) - self._h(2.0))

    def _h(self, x):
        return np.power(x, -self.q)

    def _H(self, x):
        # Antiderivative of x^-q, zero at x = 1.
        return (np.power(x, 1.0 - self.q) - 1.0) / (1.0 - self.q)

    def _Hinv(self, y):
        return np.power(1.0 + y * (1.0 - self.q), 1.0 / (1.0 - self.q))

    def ranks(self, seed: int, n: int) -> np.ndarray:
        out = np.zeros(n, np.int64)
        todo = np.arange(n)
        drawn = 0
        while todo.size:
            u = uniform01(seed, todo.size, drawn)
            drawn += todo.size
            y = self.hn + u * (self.hx1 - self.hn)
            x = self._Hinv(y)
            k = np.clip(np.floor(x + 0.5), 1, self.n)
            ok = (k - x <= self.s) | (y >= self._H(k + 0.5) - self._h(k))
            out[todo[ok]] = k[ok].astype(np.int64)
            todo = todo[~ok]
        return out


def zipf_keys(seed: int, n: int, alpha: float, universe: int, salt: int = 0x2545F4914F6CDD1D):
    """n keys whose ranks follow Zipf(alpha) over 1..universe; rank r maps to
    the key mix(r + salt), a bijection, so distinct ranks give distinct keys."""
    r = Zipf(alpha, universe).ranks(seed, n).astype(np.uint64)
    with np.errstate(over="ignore"):
        return _check_keys(mix(r + _U(salt)))


def zipf_keys_torch(seed: int, n: int, alpha: float, universe: int, device,
                    salt: int = 0x2545F4914F6CDD1D):
    """Keys of ``zipf_keys``' distribution drawn on a torch device: the same
    rejection-inversion sampler over ranks 1..universe (``Zipf``'s
    constants), its uniforms from a seeded torch generator on ``device`` (so
    not the same draws as ``zipf_keys``), rank r mapped to the key
    mix(r + salt).  Returns an int64 tensor holding the uint64 bits."""
    import torch
    z = Zipf(alpha, universe)
    q = z.q
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty(n, dtype=torch.int64, device=device)
    todo = torch.arange(n, device=device)
    while todo.numel():
        u = torch.rand(todo.numel(), dtype=torch.float64, generator=g, device=device)
        y = z.hn + u * (z.hx1 - z.hn)
        x = torch.pow(1.0 + y * (1.0 - q), 1.0 / (1.0 - q))
        k = torch.clamp(torch.floor(x + 0.5), 1, z.n)
        hk = (torch.pow(k + 0.5, 1.0 - q) - 1.0) / (1.0 - q) - torch.pow(k, -q)
        ok = (k - x <= z.s) | (y >= hk)
        out[todo[ok]] = k[ok].to(torch.int64)
        todo = todo[~ok]
    return _mix_torch(out + _i64(salt))


# --------------------------------------------------------------------------
# Values.
# --------------------------------------------------------------------------
def randn_values(seed: int, n: int, dim: int, device="cpu"):
    """n x dim float32 rows, N(0,1), from a seeded torch generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn((n, dim), generator=g, device=device, dtype=torch.float32)


def key_values(keys: np.ndarray, dim: int, salt: int = 0) -> np.ndarray:
    """Rows that depend only on (key, column, salt): uniform float32 in [-1, 1)
    with 24-bit resolution.  Exactly equal to ``key_values_torch``."""
    k = np.asarray(keys, np.uint64)[:, None]
    col = np.arange(dim, dtype=np.uint64)[None, :]
    with np.errstate(over="ignore"):
        z = mix(k ^ mix(col + _U(salt) * _U(GAMMA)))
    top = (z >> _U(40)).astype(np.int64).astype(np.float32)
    return top / np.float32(1 << 23) - np.float32(1.0)


def _i64(c: int) -> int:
    c &= 0xFFFFFFFFFFFFFFFF
    return c - (1 << 64) if c >= (1 << 63) else c


def _mix_torch(z):
    import torch

    def shr(x, s):
        return (x >> s) & ((1 << (64 - s)) - 1)

    z = (z ^ shr(z, 30)) * _i64(_M1)
    z = (z ^ shr(z, 27)) * _i64(_M2)
    return z ^ shr(z, 31)


def key_values_torch(keys, dim: int, salt: int = 0):
    """``key_values`` computed with torch int64 ops (wrapping arithmetic) on
    the keys' device; ``keys`` is an int64 tensor holding the uint64 bits."""
    import torch
    col = torch.arange(dim, dtype=torch.int64, device=keys.device)
    cm = _mix_torch(col + _i64(salt * GAMMA))
    z = _mix_torch(keys.view(-1, 1) ^ cm.view(1, -1))
    top = ((z >> 40) & 0xFFFFFF).to(torch.float32)
    return top / float(1 << 23) - 1.0


def as_i64(a: np.ndarray) -> np.ndarray:
    """View uint64 keys/scores as int64 (same bits) for torch."""
    return np.ascontiguousarray(a, np.uint64).view(np.int64)
