"""Pins of the oracle's modified Cactus lenience ([TwoTrade] App. E).

gamma* is checked against an independent high-precision bisection of eq. 17,
the modified target against its definition (its KL divergence from p, summed
over a whole vocabulary, equals delta), the small-delta limit against the
page's second-order solution (eq. 18), delta = 0 against the lossless rule
(bit for bit), and the residual weights against [ptilde - q]_+ built from the
page's ptilde."""
import math

import mpmath
import numpy as np
import pytest
from scipy import special

import oracle
from oracle import CACTUS, LOSSLESS


def _phi(g, p):
    g, p = mpmath.mpf(g), mpmath.mpf(p)
    t = g * mpmath.log(g / p)
    if g < 1:
        t += (1 - g) * mpmath.log((1 - g) / (1 - p))
    return t


def _gamma_bisect(p, delta):
    """The largest gamma in [p, 1] with Phi(gamma) <= delta, by 200 bisection
    steps at 60 significant digits."""
    mpmath.mp.dps = 60
    if _phi(1, p) <= delta:
        return 1.0
    lo, hi = mpmath.mpf(p), mpmath.mpf(1)
    for _ in range(200):
        mid = (lo + hi) / 2
        if _phi(mid, p) <= delta:
            lo = mid
        else:
            hi = mid
    return float(lo)


@pytest.mark.parametrize("p", [1e-7, 1e-3, 0.05, 0.3, 0.7, 0.99, 0.999999])
@pytest.mark.parametrize("delta", [1e-9, 1e-4, 0.01, 0.3, 1.0, 5.0])
def test_gamma_solves_eq17(orc, p, delta):
    g = orc.cactus_gamma(p, delta)
    ref = _gamma_bisect(p, delta)
    assert abs(g - ref) <= 1e-13 * max(ref, 1e-300) + 1e-300, (g, ref)
    assert p <= g <= 1.0


def test_gamma_edges(orc):
    assert orc.cactus_gamma(0.25, 0.0) == 0.25           # no budget: the target itself
    assert orc.cactus_gamma(0.25, math.log(4.0)) == 1.0  # Phi(1) = log(1/p) <= delta
    assert orc.cactus_gamma(0.0, 1.0) == 0.0
    assert orc.cactus_gamma(1.0, 1.0) == 1.0


def test_modified_target_spends_the_kl_budget(orc):
    """ptilde (gamma* on y, the rest of p scaled by (1-gamma*)/(1-p(y))) is a
    distribution whose KL divergence from p, summed over the vocabulary, is
    delta; a larger gamma would exceed it."""
    rng = np.random.default_rng(4)
    for _ in range(20):
        V = int(rng.integers(2, 300))
        p = special.softmax(rng.normal(0, 2, V))
        y = int(rng.integers(V))
        delta = float(rng.choice([1e-4, 0.02, 0.2]))
        g = orc.cactus_gamma(p[y], delta)
        if g >= 1.0:
            continue
        pt = p * (1 - g) / (1 - p[y])
        pt[y] = g
        assert abs(pt.sum() - 1.0) < 1e-12
        kl = float(np.sum(pt * np.log(pt / p)))
        assert abs(kl - delta) < 1e-10 * max(1.0, delta), (kl, delta)
        g2 = g * (1 + 1e-6)
        pt2 = p * (1 - g2) / (1 - p[y])
        pt2[y] = g2
        assert np.sum(pt2 * np.log(pt2 / p)) > delta


def test_small_delta_limit_is_the_second_order_solution(orc):
    for p in (0.01, 0.2, 0.6):
        for delta in (1e-10, 1e-8):
            g = orc.cactus_gamma(p, delta)
            taylor = math.sqrt(2 * delta * p * (1 - p))
            assert abs((g - p) / taylor - 1.0) < 1e-3


def test_acceptance_grows_with_delta(orc):
    rng = np.random.default_rng(9)
    V = 64
    lp = np.log(special.softmax(rng.normal(0, 2, V)))
    lq = np.log(special.softmax(rng.normal(0, 2, V)))
    q = np.exp(lq)
    prev = None
    for delta in (0.0, 1e-3, 0.01, 0.1, 1.0, 10.0, 50.0):
        acc = sum(q[y] * orc.accept_prob(lp[y], lq[y], CACTUS, delta) for y in range(V))
        if prev is not None:
            assert acc >= prev - 1e-15
        prev = acc
        if delta == 0.0:  # lossless: 1 - TV
            assert abs(acc - np.minimum(np.exp(lp), q).sum()) < 1e-12
    assert abs(prev - 1.0) < 1e-12  # delta >= log(1/min p): every draft accepted


def test_residual_is_the_modified_target_minus_q(orc):
    rng = np.random.default_rng(2)
    for _ in range(10):
        V = 40
        x, y = rng.normal(0, 2, V), rng.normal(0, 2, V)
        p, q = special.softmax(x), special.softmax(y)
        d = int(np.argmax(q / p))  # a token with p(d) < q(d): rejections happen
        for delta in (1e-3, 0.05, 0.5):
            g = orc.cactus_gamma(p[d], delta)
            if g >= q[d]:
                continue  # always accepted: no residual
            pt = p * (1 - g) / (1 - p[d])
            pt[d] = g
            ref = np.maximum(pt - q, 0.0)
            w = orc.residual_weights(x, y, 1.0, 1.0, CACTUS, delta, d=d)
            # differences of two probabilities: compare on the scale of p
            assert np.all(np.abs(w - ref) <= 1e-12 * p)
            assert w[d] == 0.0


def test_delta_zero_is_lossless(orc):
    import datagen
    for T, sigma in ((1.0, 0.5), (0.7, 1.0)):
        si = datagen.sample_inputs(6, 5, 2048, dtype="bf16", seed=41, sigma=sigma, T=T,
                                   ragged=True)
        args = (datagen.to_numpy_logits(si.target), datagen.to_numpy_logits(si.draft),
                si.draft_ids.numpy(), si.draft_len.numpy())
        a = orc.verify_sample(*args, T_p=T, T_q=T, mode=CACTUS, lam=0.0, seed=5)
        b = orc.verify_sample(*args, T_p=T, T_q=T, mode=LOSSLESS, seed=5)
        for k in a:
            assert np.array_equal(a[k], b[k], equal_nan=True), k
