"""Pins of the oracle's counter-based random numbers.

The mixers are pinned by published test vectors (tests/golden); the derived
uniforms and Gumbels by their distributions (closed-form moments, chi-square
goodness of fit) and by the exactness of the (2m+1)/2^53 construction.
"""
import math
import os

import numpy as np
import pytest
from scipy import stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rng_published_vectors.txt")


def _vectors():
    out = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            fn, x, y = line.split()
            out.append((fn, int(x, 16), int(y, 16)))
    return out


@pytest.mark.parametrize("fn,x,y", _vectors())
def test_published_mixer_vectors(orc, fn, x, y):
    assert getattr(orc, fn)(x) == y


def test_uniform_is_open_interval_and_exact(orc):
    for s in range(50):
        k = orc.key(s, orc.ST_SAMPLE, s * 7, s * 13, 0)
        for v in (0, 1, 2, 3, 1000, 151935):
            u = orc.uniform(k, v)
            assert 0.0 < u < 1.0
            m2 = u * 2.0 ** 53           # must be the odd integer 2m + 1
            assert m2 == int(m2) and int(m2) % 2 == 1
            assert int(m2) // 2 == orc.bits52(k, v)


def test_uniform_chi_square(orc):
    n = 40000
    k = orc.key(123, orc.ST_SAMPLE, 0, 0, 0)
    u = np.array([orc.uniform(k, v) for v in range(n)])
    counts, _ = np.histogram(u, bins=40, range=(0, 1))
    p = stats.chisquare(counts).pvalue
    assert p > 1e-4
    # the four ids that share a hash word (v = 4j .. 4j+3) are independent
    for a, b in ((0, 1), (0, 3), (1, 2)):
        pairs = np.histogram2d(u[a::4], u[b::4], bins=8, range=[[0, 1], [0, 1]])[0].ravel()
        assert stats.chisquare(pairs).pvalue > 1e-4
    top = (np.floor(u * 256)).astype(int)
    assert stats.chisquare(np.bincount(top, minlength=256)).pvalue > 1e-4
    assert abs(np.corrcoef(u[:-1], u[1:])[0, 1]) < 0.03


def test_uniform_across_keys(orc):
    # the acceptance stream uses v = 0 with a fresh key per (sequence, position)
    u = np.array([orc.uniform(orc.key(7, orc.ST_ACCEPT, b, i, 0), 0)
                  for b in range(200) for i in range(100)])
    counts, _ = np.histogram(u, bins=20, range=(0, 1))
    assert stats.chisquare(counts).pvalue > 1e-4
    ks = stats.kstest(u, "uniform").pvalue
    assert ks > 1e-4


def test_keys_differ_by_every_field(orc):
    base = (5, orc.ST_TREE, 3, 17, 2)
    k0 = orc.key(*base)
    seen = {k0}
    for i in range(5):
        f = list(base)
        f[i] += 1
        k = orc.key(*f)
        assert k not in seen
        seen.add(k)


def test_gumbel_moments(orc):
    # Gumbel(0,1): mean = Euler-Mascheroni constant, variance = pi^2/6
    k = orc.key(99, orc.ST_TREE, 0, 0, 0)
    g = np.array([orc.gumbel(k, v) for v in range(60000)])
    assert abs(g.mean() - 0.5772156649015329) < 4 * math.sqrt(math.pi ** 2 / 6 / g.size)
    assert abs(g.var() - math.pi ** 2 / 6) < 0.05
    assert stats.kstest(g, "gumbel_r").pvalue > 1e-4
