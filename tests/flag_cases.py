"""Inputs whose decisions fall within 1e-9 of their thresholds, built on the
host with the oracle (not collected as tests).

Both sides must count such a decision in `flags` and leave it out of the
bit-exact comparison.  Random inputs almost never produce one, so these are
built on purpose:
  - an acceptance test whose uniform u and probability alpha differ by a few
    1e-10: the draft token's target logit is tuned until alpha is within about
    1e-7 of u, then a low-weight logit of the same row (probability near 1e-7,
    so one fp32 step moves alpha by about 1e-13) closes the rest;
  - a Gumbel-max whose best two scores differ by a few 1e-10: a key is chosen
    whose row has two Gumbel values within 1e-3 of each other, every logit is
    0 but the runner-up's, which is set to the difference (near 1e-3, where an
    fp32 step is about 1e-10).
Logits are fp32 so that these fine steps exist.
"""
import numpy as np

import oracle

TARGET_GAP = 4e-10  # |u - alpha| or the top-two score gap aimed at


def _f32_next(x, up=True):
    return float(np.nextafter(np.float32(x), np.float32(np.inf if up else -np.inf)))


def _bisect_f32(f, lo, hi, target, increasing):
    """The float32 value x in [lo, hi] whose f(x) is closest to target, for a
    monotone f (bisection on the float32 grid)."""
    lo, hi = np.float32(lo), np.float32(hi)
    for _ in range(200):
        if _f32_next(lo) >= hi:
            break
        mid = np.float32((float(lo) + float(hi)) / 2)
        if mid <= lo or mid >= hi:
            mid = np.float32(_f32_next(lo))
        below = f(float(mid)) < target
        if below == increasing:
            lo = mid
        else:
            hi = mid
    return min((float(lo), float(hi)), key=lambda x: abs(f(x) - target))


def alpha_of(x, y, d, Tp=1.0, Tq=1.0, mode=oracle.LOSSLESS, lam=1.0):
    """The oracle's acceptance probability for draft token d."""
    Tp, Tq = oracle.f32(Tp), oracle.f32(Tq)
    lp = float(np.float64(x[d]) / Tp) - oracle.lse(x.astype(np.float64), Tp)
    lq = float(np.float64(y[d]) / Tq) - oracle.lse(y.astype(np.float64), Tq)
    return oracle.accept_prob(lp, lq, mode, oracle.f32(lam))


def near_threshold_acceptance(V, u, sign, rng, d=7, w=11):
    """fp32 rows (x, y) of a target and drafter with |u - alpha(d)| about
    TARGET_GAP, alpha above u when sign > 0 (accepted) and below otherwise."""
    x = rng.standard_normal(V).astype(np.float32)
    y = (x + 0.5 * rng.standard_normal(V)).astype(np.float32)
    goal = u + sign * TARGET_GAP
    x[w] = -20.0

    def a_xd(v):
        x[d] = v
        return alpha_of(x, y, d)

    # coarse: the smallest x_d with alpha >= goal (alpha grows with x_d)
    xd = _bisect_f32(a_xd, -30.0, 30.0, goal, True)
    x[d] = xd
    while alpha_of(x, y, d) < goal:
        x[d] = _f32_next(x[d])

    # fine: raise the low-weight logit x_w until alpha comes down to the goal
    def a_xw(v):
        x[w] = v
        return alpha_of(x, y, d)

    x[w] = _bisect_f32(a_xw, -20.0, -2.0, goal, False)
    return x, y, abs(alpha_of(x, y, d) - u)


def near_tie_key(make_key, V, start=0, tries=200000, gap_max=1e-3):
    """The first p >= start whose key make_key(p) gives a row (ids 0..V-1) with
    its two largest Gumbel values within gap_max; returns (p, a, b): the best
    id a and the runner-up b."""
    for p in range(start, start + tries):
        k = make_key(p)
        g = np.array([oracle.gumbel(k, v) for v in range(V)]) if V <= 64 else None
        if g is None:
            u, top = oracle.row_uniforms(k, V)
            g = -np.log(-np.log(u))
        o = np.argsort(-g, kind="stable")
        if g[o[0]] - g[o[1]] < gap_max:
            a, b = int(o[0]), int(o[1])
            ga, gb = oracle.gumbel(k, a), oracle.gumbel(k, b)
            if ga >= gb:
                return p, a, b
            return p, b, a
    raise RuntimeError("no near tie found")


def near_tie_row(k, V, a, b, T, sign):
    """An fp32 row, 0 everywhere but at the runner-up b, whose Gumbel-max
    scores x/T + G of ids a and b differ by about TARGET_GAP: b ahead when
    sign > 0."""
    T = oracle.f32(T)
    ga, gb = oracle.gumbel(k, a), oracle.gumbel(k, b)
    x = np.zeros(V, np.float32)

    def diff(v):  # score(b) - score(a)
        return float(np.float64(np.float32(v)) / T) + gb - ga

    goal = sign * TARGET_GAP
    x[b] = _bisect_f32(diff, 0.0, 1.0, goal, True)
    return x, abs(diff(x[b]))
