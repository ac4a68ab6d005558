"""The near-threshold inputs of flag_cases.py do what they are built for: the
oracle counts each crafted decision in `flags`, and the crafted decisions come
out the way they were aimed (accepted / rejected; the intended Gumbel winner).
The GPU tests in test_gpu_flags.py reuse the same inputs."""
import numpy as np

import oracle
from flag_cases import TARGET_GAP, near_threshold_acceptance, near_tie_key, near_tie_row

V = 4096


def test_crafted_acceptance_is_flagged(orc):
    rng = np.random.default_rng(3)
    for b, sign in ((0, 1), (1, -1)):
        pos = 40
        u = orc.uniform(orc.key(11, orc.ST_ACCEPT, b, pos, 0), 0)
        x, y, gap = near_threshold_acceptance(V, u, sign, rng)
        assert gap < 1e-9 and abs(gap - TARGET_GAP) < 2e-10
        # a batch of two with the crafted row pair at sequence b (the
        # sequence index enters the key) and a random one at the other
        tg = np.zeros((2, 2, V), np.float32)
        dr = np.zeros((2, 1, V), np.float32)
        tg[b, 0], tg[b, 1], dr[b, 0] = x, rng.standard_normal(V), y
        other = 1 - b
        tg[other] = rng.standard_normal((2, V))
        dr[other, 0] = tg[other, 0] + 0.5 * rng.standard_normal(V)
        ids = np.array([[7], [7]], np.int32)
        r = orc.verify_sample(tg, dr, ids, seed=11, pos_base=np.array([40, 40]), want_tv=False)
        assert r["flags"][b] == 1
        assert r["accept_len"][b] == (1 if sign > 0 else 0)


def test_crafted_gumbel_tie_is_flagged(orc):
    for sign in (1, -1):
        p, a, b = near_tie_key(lambda q: orc.key(5, orc.ST_SAMPLE, 0, q, 0), V,
                               start=1000 if sign > 0 else 5000)
        k = orc.key(5, orc.ST_SAMPLE, 0, p, 0)
        x, gap = near_tie_row(k, V, a, b, 1.0, sign)
        assert gap < 1e-9
        win, g = orc.gumbel_argmax(x.astype(np.float64), k)
        assert g < 1e-9 and win == (b if sign > 0 else a)
        # as the bonus draw of a call with no draft tokens
        r = orc.verify_sample(x[None, None], np.zeros((1, 0, V), np.float32),
                              np.zeros((1, 0), np.int32), seed=5, pos_base=np.array([p]),
                              want_tv=False)
        assert r["flags"][0] == 1 and r["next_token"][0] == win
