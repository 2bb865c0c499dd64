"""The seeded input generators (CPU only)."""
import numpy as np
import pytest
import torch

import workloads as wl


def test_unique_keys_are_distinct_and_seeded():
    a = wl.unique_keys(1, 200000)
    assert np.unique(a).size == a.size
    assert np.array_equal(a, wl.unique_keys(1, 200000))
    assert np.array_equal(a[1000:2000], wl.unique_keys(1, 1000, start=1000))
    assert np.intersect1d(a, wl.unique_keys(2, 200000)).size == 0


def test_zipf_matches_pmf():
    """Rejection-inversion reproduces P(r) ~ r^-alpha on a small universe."""
    for alpha, n in ((1.05, 50), (1.5, 20), (0.8, 30)):
        r = wl.Zipf(alpha, n).ranks(7, 400000)
        assert r.min() >= 1 and r.max() <= n
        p = np.arange(1, n + 1, dtype=np.float64) ** -alpha
        p /= p.sum()
        emp = np.bincount(r, minlength=n + 1)[1:] / r.size
        sd = np.sqrt(p * (1 - p) / r.size)
        assert np.all(np.abs(emp - p) < 5 * sd + 1e-12), (alpha, np.abs(emp - p) / sd)


def test_key_values_numpy_equals_torch():
    k = wl.unique_keys(3, 5000)
    a = wl.key_values(k, 7, salt=5)
    b = wl.key_values_torch(torch.from_numpy(wl.as_i64(k)), 7, salt=5).numpy()
    assert np.array_equal(a, b)
    assert a.min() >= -1 and a.max() < 1


def test_hit_mix_fraction():
    res = wl.unique_keys(4, 10000)
    keys, drawn = wl.hit_mix(5, res, 6, 20000, 0.8)
    assert drawn.sum() == 16000
    assert np.isin(keys[drawn], res).all()
    assert not np.isin(keys[~drawn], res).any()


@pytest.mark.parametrize("alpha", [0.5, 0.99, 1.25])
def test_zipf_torch_sampler_distribution(alpha):
    """The device sampler draws ranks with the Zipf(alpha) probabilities
    r^-alpha / sum(r^-alpha) over 1..U (U = 1000, exact): each of the top
    ranks' frequency within 5 standard deviations, Pearson's chi-square over
    all U ranks within 6 standard deviations of its mean (U - 1 degrees of
    freedom), and rank r maps to the host sampler's key for r."""
    import torch
    U, n = 1000, 1 << 20
    keys = wl.zipf_keys_torch(7, n, alpha, U, "cpu").numpy().view(np.uint64)
    ranks = np.arange(1, U + 1, dtype=np.uint64)
    key_of = wl.mix(ranks + np.uint64(0x2545F4914F6CDD1D))
    pos = {int(k): i for i, k in enumerate(key_of)}
    idx = np.array([pos[int(k)] for k in keys])  # every key is some rank's key
    counts = np.bincount(idx, minlength=U)
    p = ranks.astype(np.float64) ** -alpha
    p /= p.sum()
    emp = counts / n
    for r in range(20):
        sd = np.sqrt(p[r] * (1 - p[r]) / n)
        assert abs(emp[r] - p[r]) < 5 * sd, (r + 1, emp[r], p[r])
    chi2 = float((((counts - n * p) ** 2) / (n * p)).sum())
    assert chi2 < (U - 1) + 6 * np.sqrt(2 * (U - 1)), chi2
