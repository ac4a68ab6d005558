"""Pins of the oracle's per-row primitives against library routines and
closed forms: log-sum-exp, argmax tie-break, total variation, Gumbel-max."""
import math

import numpy as np
import pytest
from scipy import special, stats


@pytest.mark.parametrize("T", [0.3, 0.7, 1.0, 2.5])
def test_lse_matches_scipy(orc, T):
    rng = np.random.default_rng(1)
    for V in (1, 2, 7, 1000, 32000):
        x = rng.normal(0, 2, V)
        assert orc.lse(x, T) == pytest.approx(special.logsumexp(x / T), rel=1e-14, abs=1e-13)


def test_lse_closed_forms(orc):
    V = 4096
    assert orc.lse(np.full(V, 3.0), 0.5) == pytest.approx(6.0 + math.log(V), rel=1e-15)
    # two entries: log(e^a + e^b)
    assert orc.lse(np.array([1.0, -2.0]), 1.0) == pytest.approx(
        1.0 + math.log1p(math.exp(-3.0)), rel=1e-15)
    # huge logits must not overflow
    assert orc.lse(np.array([1e4, 1e4]), 1.0) == pytest.approx(1e4 + math.log(2), rel=1e-15)


def test_argmax_lowest_index_on_ties(orc):
    x = np.array([0.0, 5.0, 1.0, 5.0, 5.0, -1.0])
    assert orc.argmax(x) == 1 == int(np.argmax(x))
    rng = np.random.default_rng(2)
    for _ in range(200):
        # bf16-like coarse values produce frequent exact ties
        x = np.round(rng.normal(0, 2, 300) * 4) / 4
        assert orc.argmax(x) == int(np.argmax(x))


def test_tv_is_half_l1(orc):
    # [TwoTrade] eq. (2): D_TV = 1/2 sum |p - q|, against the oracle's 1 - sum min
    rng = np.random.default_rng(3)
    for _ in range(20):
        V = int(rng.integers(2, 500))
        x, y = rng.normal(0, 2, V), rng.normal(0, 2, V)
        Tp, Tq = rng.uniform(0.5, 1.5, 2)
        p = special.softmax(x / Tp)
        q = special.softmax(y / Tq)
        assert orc.tv(x, y, Tp, Tq) == pytest.approx(0.5 * np.abs(p - q).sum(), abs=1e-14)
    x = rng.normal(0, 2, 50)
    assert abs(orc.tv(x, x, 1.0, 1.0)) < 1e-15


def test_gumbel_argmax_law(orc):
    # [SPOT] eqs. (5)-(7): Pr[argmax(l + G) = u] = softmax(l)_u
    score = np.array([0.3, -1.0, 1.2, 0.0, -np.inf, 0.7])
    n = 30000
    counts = np.zeros(score.size)
    for s in range(n):
        idx, gap = orc.gumbel_argmax(score, orc.key(s, orc.ST_SAMPLE, 0, 0, 0))
        counts[idx] += 1
        assert gap > 0
    assert counts[4] == 0  # zero weight is never drawn
    p = special.softmax(np.where(np.isinf(score), -1e300, score))
    keep = p > 0
    assert stats.chisquare(counts[keep], n * p[keep]).pvalue > 1e-4


def test_gumbel_argmax_temperature_law(orc):
    # sampling softmax(x / T) through the identity at T = 0.5
    x = np.array([1.0, 0.5, 0.0, -0.5])
    T = 0.5
    n = 20000
    counts = np.zeros(4)
    for s in range(n):
        counts[orc.gumbel_argmax(x / T, orc.key(s, orc.ST_DRAFT, 1, 2, 3))[0]] += 1
    assert stats.chisquare(counts, n * special.softmax(x / T)).pvalue > 1e-4


def test_gumbel_coupling_bound(orc):
    # [SPOT] §4.3: two rows under shared noise agree with probability at least
    # (1 - delta) / (1 + delta), delta = TV distance of their laws
    rng = np.random.default_rng(4)
    for trial in range(4):
        x = rng.normal(0, 1, 12)
        y = x + rng.normal(0, 0.6, 12)
        delta = 0.5 * np.abs(special.softmax(x) - special.softmax(y)).sum()
        n = 6000
        agree = 0
        for s in range(n):
            k = orc.key(1000 * trial + s, orc.ST_TREE, 0, 0, 0)
            agree += orc.gumbel_argmax(x, k)[0] == orc.gumbel_argmax(y, k)[0]
        bound = (1 - delta) / (1 + delta)
        assert agree / n > bound - 4 * math.sqrt(bound * (1 - bound) / n)
