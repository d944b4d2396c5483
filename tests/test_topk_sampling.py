"""The top-k kernel's long-window threshold, checked as a statistical design
claim on the CPU (numpy; no kernel code involved).

A window of L values longer than the candidate capacity C is sampled with
stride S = ceil(L / C); the (k/S + 5 sqrt(k/S) + 16)-th largest sample key
(the rank computed in f32 and truncated, as the kernel does), rounded down
to its 24-bit radix bin, is a lower threshold; the values at or above it are
the candidates, and the fast path needs k <= #candidates <= C.  The sample
holds about k/S values above the true k-th, give or take sqrt(k/S), so
about rank * S values should pass, several standard deviations from both
bounds for independent values -- this test measures that over the shapes the
kernel meets (decode windows of 131072, prefill windows up to 65536, k 512
and 2048) and a few value distributions.
"""
import numpy as np
import pytest

CAP = 8192


def order_keys(x):
    u = (x.astype(np.float32) + np.float32(0.0)).view(np.uint32)
    return np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)


def candidates(vals, k):
    L = vals.size
    S = -(-L // CAP)
    keys = order_keys(vals)
    sample = keys[::S]
    kS = np.float32(k) / np.float32(S)
    rank = min(int(kS + np.float32(5.0) * np.sqrt(kS)) + 16, sample.size)
    t = np.sort(sample)[::-1][rank - 1] & np.uint32(0xFFFFFF00)
    return int(np.count_nonzero(keys >= t)), rank * S


DISTS = {
    "normal": lambda rng, n: rng.normal(size=n),
    "laplace": lambda rng, n: rng.laplace(size=n),
    "uniform": lambda rng, n: rng.uniform(-1, 1, size=n),
    "relu_sum": lambda rng, n: np.maximum(rng.normal(size=(n, 4)), 0).sum(axis=1) - 1.0,  # skewed, like the logits
}


@pytest.mark.parametrize("dist", sorted(DISTS))
@pytest.mark.parametrize("L,k", [(131072, 2048), (131072, 512), (65536, 2048), (16384, 2048), (8200, 2048)])
def test_candidate_count_within_bounds(dist, L, k):
    rng = np.random.default_rng(L + k)
    counts, expect = [], None
    for _ in range(20):
        n, expect = candidates(DISTS[dist](rng, L).astype(np.float32), k)
        counts.append(n)
    counts = np.array(counts)
    assert counts.min() >= k, (dist, L, k, counts.min())
    assert counts.max() <= CAP, (dist, L, k, counts.max())
    # the spread leaves room on both sides: at least 3 standard deviations
    # of the observed candidate counts (which also carry the spread of the
    # threshold sample's own gaps)
    sd = max(counts.std(), 1.0)
    assert counts.mean() - 3 * sd >= k and counts.mean() + 4 * sd <= CAP, (dist, L, k, counts.mean(), sd)
    # and the mean lands near the design's rank * S
    assert 0.6 * expect <= counts.mean() <= 1.6 * expect, (dist, L, k, counts.mean(), expect)


@pytest.mark.parametrize("L,k", [(131072, 2048), (131072, 512), (65536, 2048), (16384, 2048), (8200, 2048),
                                 (1 << 20, 2048), (1 << 20, 512)])
def test_fallback_probability(L, k):
    """The fast path misses only if the stride sample holds at least `rank`
    of the window's k largest values: for independent values that count is
    Binomial(k, 1/S), and the rank leaves it below 1e-6 (the exact fallback
    keeps the result right either way)."""
    from scipy.stats import binom
    S = -(-L // CAP)
    kS = np.float32(k) / np.float32(S)
    rank = int(kS + np.float32(5.0) * np.sqrt(kS)) + 16
    assert binom.sf(rank - 1, k, 1.0 / S) < 1e-6, (L, k, S, rank)
    assert rank * S <= CAP, (L, k, S, rank)  # the expected candidates fit the shared-memory capacity
