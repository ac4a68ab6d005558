"""Exact (enumeration) pins of the oracle's acceptance and residual rules.

Tiny vocabularies (V <= 5) and drafts (K <= 3): every draft sequence is
enumerated with its proposal probability, the uniforms are integrated out
analytically (Pr[accept] = alpha), and the law of the emitted tokens is
compared with the target's autoregressive chain rule to 1e-12.
"""
import itertools

import numpy as np
import pytest
from scipy import special

LOSSLESS, RATIO, LINEAR = 0, 1, 2


class ToyAR:
    """A toy autoregressive target: logits for every prefix from a seeded hash."""

    def __init__(self, V, seed, scale=1.5):
        self.V, self.seed, self.scale = V, seed, scale
        self._cache = {}

    def logits(self, prefix):
        prefix = tuple(prefix)
        if prefix not in self._cache:
            rng = np.random.default_rng([self.seed, len(prefix)] + list(prefix))
            self._cache[prefix] = rng.normal(0, self.scale, self.V)
        return self._cache[prefix]

    def probs(self, prefix, T):
        return special.softmax(self.logits(prefix) / T)


def emitted_law(orc, target, drafter, K, V, Tp, Tq, mode, lam):
    """Law over V^(K+1) of the emitted block continued by the target model."""
    law = np.zeros((V,) * (K + 1))
    for d in itertools.product(range(V), repeat=K):
        # proposal probability of this draft (drafter may depend on d_<i)
        ys = [drafter(d[:i]) for i in range(K)]
        qs = [special.softmax(y / Tq) for y in ys]
        wdraft = np.prod([qs[i][d[i]] for i in range(K)])
        if wdraft == 0:
            continue
        xs = [target.logits(d[:i]) for i in range(K + 1)]
        reach = 1.0
        for h in range(K + 1):
            if h < K:
                lp = xs[h][d[h]] / Tp - orc.lse(xs[h], Tp)
                lq = ys[h][d[h]] / Tq - orc.lse(ys[h], Tq)
                alpha = orc.accept_prob(lp, lq, mode, lam)
                w = orc.residual_weights(xs[h], ys[h], Tp, Tq, mode, lam)
                rej = reach * (1.0 - alpha)
                if rej > 0 and w.sum() > 0:
                    corr = w / w.sum()
                else:
                    corr = np.zeros(V)
            else:
                rej = reach
                corr = special.softmax(xs[K] / Tp)
            for c in range(V):
                if rej * corr[c] == 0:
                    continue
                block = d[:h] + (c,)
                tail = list(itertools.product(range(V), repeat=K - h))
                for t in tail:
                    pr = wdraft * rej * corr[c]
                    seq = block + t
                    for j in range(h + 1, K + 1):
                        pr *= target.probs(seq[:j], Tp)[seq[j]]
                    law[seq] += pr
            if h < K:
                reach *= alpha
    return law


def chain_rule(target, K, V, Tp, mix=None):
    law = np.zeros((V,) * (K + 1))
    for seq in itertools.product(range(V), repeat=K + 1):
        pr = 1.0
        for j in range(K + 1):
            p = target.probs(seq[:j], Tp)
            if mix is not None:
                p = mix(seq[:j], p)
            pr *= p[seq[j]]
        law[seq] = pr
    return law


@pytest.mark.parametrize("K,V,Tp,Tq,ar_drafter", [
    (1, 5, 1.0, 1.0, False), (2, 4, 0.7, 1.0, False), (3, 3, 1.0, 0.8, False),
    (2, 4, 1.0, 1.0, True), (3, 3, 1.3, 1.3, True)])
def test_lossless_reproduces_target_law(orc, K, V, Tp, Tq, ar_drafter):
    # [PackedSS] Lemma B.3 / Thm 3.3; [SPOT] Prop. 3: the emitted tokens follow
    # the target's chain rule exactly, for any proposal.
    target = ToyAR(V, seed=11 + K)
    rng = np.random.default_rng(5)
    fixed = [rng.normal(0, 1.5, V) for _ in range(K)]
    drafter = (lambda pre: ToyAR(V, 99).logits(pre)) if ar_drafter else \
        (lambda pre: fixed[len(pre)])
    law = emitted_law(orc, target, drafter, K, V, Tp, Tq, LOSSLESS, 1.0)
    ref = chain_rule(target, K, V, Tp)
    assert np.abs(law - ref).max() < 1e-12
    assert abs(law.sum() - 1.0) < 1e-12


def test_lossless_with_point_mass_and_disjoint_support(orc):
    # Lemma B.3 needs no full support: q putting all mass on one token, and p,q
    # with disjoint high-mass regions, still give the exact law.
    V, K = 4, 2
    target = ToyAR(V, seed=3)
    spike = np.array([40.0, -40.0, -40.0, -40.0])
    law = emitted_law(orc, target, lambda pre: spike, K, V, 1.0, 1.0, LOSSLESS, 1.0)
    assert np.abs(law - chain_rule(target, K, V, 1.0)).max() < 1e-12


@pytest.mark.parametrize("Tp,Tq", [(1.0, 1.0), (0.7, 1.2)])
def test_acceptance_is_one_minus_tv(orc, Tp, Tq):
    # [TwoTrade] eq. (1): sum_d q(d) min{1, p(d)/q(d)} = 1 - D_TV(p, q), with
    # D_TV = 1/2 sum |p - q| (eq. (2)).
    rng = np.random.default_rng(6)
    for _ in range(30):
        V = int(rng.integers(2, 40))
        x, y = rng.normal(0, 2, V), rng.normal(0, 2, V)
        p, q = special.softmax(x / Tp), special.softmax(y / Tq)
        Lp, Lq = orc.lse(x, Tp), orc.lse(y, Tq)
        acc = sum(q[d] * orc.accept_prob(x[d] / Tp - Lp, y[d] / Tq - Lq) for d in range(V))
        assert acc == pytest.approx(1.0 - 0.5 * np.abs(p - q).sum(), abs=1e-13)


@pytest.mark.parametrize("mu", [0.0, 0.25, 0.5, 0.875, 1.0])
def test_linear_lenience_theorem(orc, mu):
    # [TwoTrade] Thm 1 / eq. (5): with ptilde = (1-mu)p + mu q the acceptance is
    # 1 - (1-mu) D_TV(p,q) and the emitted token follows ptilde exactly.
    rng = np.random.default_rng(7)
    for _ in range(20):
        V = int(rng.integers(2, 30))
        x, y = rng.normal(0, 2, V), rng.normal(0, 2, V)
        p, q = special.softmax(x), special.softmax(y)
        Lp, Lq = orc.lse(x, 1.0), orc.lse(y, 1.0)
        alpha = np.array([orc.accept_prob(x[d] - Lp, y[d] - Lq, LINEAR, mu) for d in range(V)])
        beta = float((q * alpha).sum())
        tvd = 0.5 * np.abs(p - q).sum()
        assert beta == pytest.approx(1.0 - (1.0 - mu) * tvd, abs=1e-13)
        w = orc.residual_weights(x, y, 1.0, 1.0, LINEAR, mu)
        out = q * alpha + ((1.0 - beta) * w / w.sum() if w.sum() > 0 else 0.0)
        assert np.abs(out - ((1 - mu) * p + mu * q)).max() < 1e-13


@pytest.mark.parametrize("lam", [1.0, 2.0, 4.0, 8.0])
def test_ratio_lenience_acceptance(orc, lam):
    # accept w.p. min{1, lam p/q}: sum_d q(d) alpha(d) = sum_v min{q_v, lam p_v}
    rng = np.random.default_rng(8)
    for _ in range(20):
        V = int(rng.integers(2, 30))
        x, y = rng.normal(0, 2, V), rng.normal(0, 2, V)
        p, q = special.softmax(x), special.softmax(y)
        Lp, Lq = orc.lse(x, 1.0), orc.lse(y, 1.0)
        acc = sum(q[d] * orc.accept_prob(x[d] - Lp, y[d] - Lq, RATIO, lam) for d in range(V))
        assert acc == pytest.approx(np.minimum(q, lam * p).sum(), abs=1e-13)


def test_ratio_one_is_lossless_law(orc):
    V, K = 4, 2
    target = ToyAR(V, seed=31)
    dr = ToyAR(V, seed=32)
    a = emitted_law(orc, target, dr.logits, K, V, 1.0, 1.0, RATIO, 1.0)
    b = emitted_law(orc, target, dr.logits, K, V, 1.0, 1.0, LOSSLESS, 1.0)
    assert np.array_equal(a, b)
