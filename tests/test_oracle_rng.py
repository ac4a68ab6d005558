"""Pins of the oracle's counter-based random numbers.

The mixer is pinned by published test vectors (tests/golden); the skip
thresholds by an independent exact-integer computation; the top-id process by
its binomial law per block of 256 ids; the uniforms and Gumbels by their
distributions (closed-form moments, chi-square goodness of fit) and by the
exactness of the (2m+1)/2^53 construction.
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


def test_skip_thresholds_are_exact(orc):
    # C_g = ceil(2^64 (255/256)^g), here with Python's exact integers
    for g in range(1, 257):
        exact = -((-(2**64) * 255**g) // 256**g)
        assert orc.skip_threshold(g) == exact, g


def test_uniform_is_open_interval_and_exact(orc):
    for s in range(40):
        k = orc.key(s, orc.ST_SAMPLE, s * 7, s * 13, 0)
        for v in (0, 1, 2, 3, 255, 256, 1000, 151935):
            u = orc.uniform(k, v)
            assert 0.0 < u < 1.0
            m = orc.fine52(k, v)
            assert 0 <= m < 2**52
            w = (2 * m + 1) * 2.0**-53
            if orc.is_top(k, v):
                assert u >= 255 / 256 and 1.0 - u == pytest.approx((1.0 - w) / 256, abs=2**-53)
            else:
                assert u < 255 / 256 and u == w * (255 / 256)


def test_top_ids_are_bernoulli_per_block(orc):
    # counts per block of 256 ids ~ Binomial(256, 1/256); offsets uniform
    counts, offsets = [], []
    for s in range(120):
        k = orc.key(1000 + s, orc.ST_TREE, s, 3 * s, 0)
        _, top = orc.row_uniforms(k, 256 * 40)
        t = top.reshape(40, 256)
        counts.extend(t.sum(1).tolist())
        offsets.extend(np.nonzero(t)[1].tolist())
    counts = np.array(counts)
    n = counts.size
    p = [stats.binom.pmf(c, 256, 1 / 256) for c in range(3)]
    p.append(1.0 - sum(p))
    obs = [np.sum(counts == 0), np.sum(counts == 1), np.sum(counts == 2), np.sum(counts >= 3)]
    assert stats.chisquare(obs, np.array(p) * n).pvalue > 1e-4
    assert abs(counts.mean() - 1.0) < 4 * math.sqrt(255 / 256 / n)
    assert stats.chisquare(np.bincount(np.array(offsets) // 16, minlength=16)).pvalue > 1e-4


def test_uniform_chi_square(orc):
    n = 60000
    k = orc.key(123, orc.ST_SAMPLE, 0, 0, 0)
    u, top = orc.row_uniforms(k, n)
    counts, _ = np.histogram(u, bins=40, range=(0, 1))
    assert stats.chisquare(counts).pvalue > 1e-4
    # the top bucket [255/256, 1) holds exactly the top ids, and a fine
    # histogram inside it is flat
    assert np.array_equal(u >= 255 / 256, top)
    inner = (u[top] - 255 / 256) * 256
    assert stats.chisquare(np.histogram(inner, bins=8, range=(0, 1))[0]).pvalue > 1e-4
    # neighbours (inside and across blocks) are independent
    for lag in (1, 2, 255, 256):
        pairs = np.histogram2d(u[:-lag], u[lag:], bins=8, range=[[0, 1], [0, 1]])[0].ravel()
        assert stats.chisquare(pairs).pvalue > 1e-4
    assert abs(np.corrcoef(u[:-1], u[1:])[0, 1]) < 0.03


def test_uniform_across_keys(orc):
    # the acceptance stream uses v = 0 with a fresh key per (sequence, position)
    u = np.array([orc.uniform(orc.key(7, orc.ST_ACCEPT, b, i, 0), 0)
                  for b in range(200) for i in range(100)])
    counts, _ = np.histogram(u, bins=20, range=(0, 1))
    assert stats.chisquare(counts).pvalue > 1e-4
    assert stats.kstest(u, "uniform").pvalue > 1e-4


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
    # the upper tail comes from the top ids: P(G > 5.5414) = 1/256
    assert abs(np.mean(g > -math.log(-math.log(255 / 256))) - 1 / 256) < 4 * math.sqrt(1 / 256 / g.size)


FROZEN = os.path.join(os.path.dirname(__file__), "golden", "rng_frozen_vectors.txt")


def _frozen():
    rows, key = [], None
    for line in open(FROZEN):
        f = line.split("#")[0].split()
        if not f:
            continue
        if f[0] == "key":
            key = tuple(int(x) for x in f[1:6]) + (int(f[6], 16),)
        else:
            rows.append((key, int(f[1]), int(f[2]), int(f[3], 16), float.fromhex(f[4]),
                         float.fromhex(f[5])))
    return rows


def test_frozen_vectors_cover_the_layout():
    rows = _frozen()
    assert len(rows) >= 32
    assert {k[1] for k, *_ in rows} == {1, 2, 3, 4}       # every stream
    assert any(top for _, v, top, *_ in rows if v >= 151808)  # a top id in the last block
    assert sum(top for _, _, top, *_ in rows) >= 9           # top ids of every key
    assert any(k[4] >= 2**32 for k, *_ in rows) and any(k[3] >= 2**40 for k, *_ in rows)


def test_oracle_matches_frozen_vectors(orc):
    """The oracle's key, top flag, fine bits, uniform and Gumbel value, bit for
    bit, against values frozen from an earlier build of the same layout."""
    for (seed, st, seq, pos, it, k), v, top, m, u, g in _frozen():
        assert orc.key(seed, st, seq, pos, it) == k
        assert int(orc.is_top(k, v)) == top, (k, v)
        assert orc.fine52(k, v) == m, (k, v)
        assert orc.uniform(k, v) == u, (k, v)
        assert orc.gumbel(k, v) == g, (k, v)
