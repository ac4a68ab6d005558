"""Pins of the oracle's Packed-SS step with top-k truncated distributions
([PackedSS] §3.2, last paragraph; Alg. 2; Thm. 3.3).

- The top-k selection equals a lexicographic sort (logit descending, id
  ascending) of the row, ties included.
- k = V keeps every entry: the step is the untruncated Alg. 2 step, given the
  full stored Q as lists.
- k = 1 on both sides makes both distributions point masses at the argmax:
  the step is the greedy Alg. 1 step.
- Law of one step (Thm. 3.3 with the truncated target): with the draft drawn
  from the truncated Q, the first committed token follows the truncated
  target; the proposals follow the truncated drafter distribution.
- Stored lists: ids in the order of the selection, probabilities summing to
  1, every next-draft token in its list.
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle


def lex_topk(x, k):
    return np.lexsort((np.arange(len(x)), -x))[:k]


@pytest.mark.parametrize("seed", range(4))
def test_topk_is_a_lexicographic_sort(orc, seed):
    rng = np.random.default_rng(seed)
    for V, k in [(1, 1), (7, 3), (50, 50), (300, 20), (2000, 64)]:
        for x in (rng.normal(0, 2, V), rng.integers(0, 4, V).astype(np.float64),
                  np.full(V, 1.5)):
            assert list(orc.topk(x, k)) == list(lex_topk(x, k))


def _prev_lists(prev_rows, T, k):
    """Top-k lists (ids, fp32 probabilities) of the previous drafter rows."""
    B, W, V = prev_rows.shape
    ids = np.empty((B, W, k), np.int32)
    probs = np.empty((B, W, k), np.float32)
    for b in range(B):
        for j in range(W):
            y = prev_rows[b, j].astype(np.float64)
            s = lex_topk(y, k)
            ids[b, j] = s
            probs[b, j] = special.softmax(y[s] / np.float64(np.float32(T)))
    return ids, probs


def _draw(ids, probs, rng):
    return int(ids[np.searchsorted(np.cumsum(probs.astype(np.float64)), rng.random() * probs.astype(np.float64).sum())])


@pytest.mark.parametrize("T", [0.7, 1.0])
def test_full_k_is_the_untruncated_step(orc, T):
    rng = np.random.default_rng(11)
    B, K, W, V = 24, 6, 6, 40
    logits = rng.normal(0, 2, (B, K + W, V)).astype(np.float32)
    prev_rows = rng.normal(0, 2, (B, W, V)).astype(np.float32)
    off = rng.integers(0, 3, B).astype(np.int32)
    n = np.minimum(rng.integers(0, K, B), W - off).astype(np.int32)
    qi, qp = _prev_lists(prev_rows, T, V)
    drafts = np.zeros((B, K - 1), np.int32)
    qd = np.ones((B, K - 1), np.float32)
    for b in range(B):
        for i in range(n[b]):
            # the draft equals the row's argmax half the time, so that both
            # acceptances and rejections occur
            row = logits[b, i].astype(np.float64)
            d = int(np.argmax(row)) if rng.random() < 0.5 else _draw(qi[b, off[b] + i], qp[b, off[b] + i], rng)
            drafts[b, i] = d
            qd[b, i] = qp[b, off[b] + i][list(qi[b, off[b] + i]).index(d)]
    ref = orc.packed_step(logits, K, W, drafts, n, prev_q_at_draft=qd, prev_draft_logits=prev_rows,
                          prev_q_offset=off, T=T, seed=5, it=2)
    out = orc.packed_topk_step(logits, K, W, V, V, drafts, n, qi, qp, off, T, seed=5, it=2)
    ok = (ref["flags"] == 0) & (out["flags"] == 0)
    assert ok.sum() >= B - 1
    for key in ("accept_len", "commit_len", "committed", "next_draft", "next_len"):
        assert np.array_equal(out[key][ok], ref[key][ok]), key
    m = out["next_draft"][ok] >= 0
    np.testing.assert_allclose(out["next_q_at_draft"][ok][m], ref["next_q_at_draft"][ok][m],
                               rtol=1e-12)
    assert ref["accept_len"].max() >= 1 and (ref["accept_len"] < n).any()


def test_k1_is_the_greedy_step(orc):
    rng = np.random.default_rng(12)
    B, K, W, V = 30, 5, 5, 25
    logits = rng.normal(0, 2, (B, K + W, V)).astype(np.float32)
    prev_rows = rng.normal(0, 2, (B, W, V)).astype(np.float32)
    for b in range(B):  # make some drafts right
        for i in range(K - 1):
            if rng.random() < 0.7:
                prev_rows[b, i] = logits[b, i]
    off = np.zeros(B, np.int32)
    n = rng.integers(0, K, B).astype(np.int32)
    qi, qp = _prev_lists(prev_rows, 1.0, 1)
    drafts = qi[:, :K - 1, 0].copy()
    ref = orc.packed_step(logits, K, W, drafts, n, T=0.0)
    out = orc.packed_topk_step(logits, K, W, 1, 1, drafts, n, qi, qp, off, 1.0, seed=3)
    for key in ("accept_len", "commit_len", "committed", "next_draft", "next_len"):
        assert np.array_equal(out[key], ref[key]), key
    assert np.all(out["q_probs"] == 1.0)
    assert 0 < ref["accept_len"].mean() < K - 1


@pytest.mark.parametrize("kp,kq", [(3, 2), (2, 4), (6, 6)])
def test_law_of_one_step(orc, kp, kq):
    """One draft position: C_0 = d if accepted, else the correction.  With d
    drawn from the truncated Q of its stored list, C_0 follows the truncated
    target p~ of verify row 0, whose support may differ from Q's."""
    rng = np.random.default_rng(100 + kp * 10 + kq)
    V, K, W, N, T = 6, 2, 2, 30000, 1.0
    x = np.array([1.2, 0.3, 1.0, -0.4, 0.9, 0.0], np.float32)     # target, verify row 0
    yprev = np.array([0.1, 1.5, 1.1, 0.2, -1.0, 0.6], np.float32)  # stored drafter row
    row1 = rng.normal(0, 1, V).astype(np.float32)
    logits = np.broadcast_to(np.stack([x, row1, row1, row1])[None], (N, K + W, V)).copy()
    qi1, qp1 = _prev_lists(yprev[None, None], T, kq)
    qi = np.broadcast_to(qi1, (N, W, kq)).copy()
    qp = np.broadcast_to(qp1, (N, W, kq)).copy()
    cdf = np.cumsum(qp1[0, 0].astype(np.float64))
    drafts = qi1[0, 0][np.minimum(np.searchsorted(cdf, rng.random(N) * cdf[-1]), kq - 1)]
    out = orc.packed_topk_step(logits, K, W, kp, kq, drafts[:, None], np.ones(N, np.int32), qi,
                               qp, np.zeros(N, np.int32), T, seed=9)
    assert np.all(out["flags"] == 0)
    c0 = out["committed"][:, 0]
    s = lex_topk(x.astype(np.float64), kp)
    p = np.zeros(V)
    p[s] = special.softmax(x.astype(np.float64)[s] / T)
    counts = np.bincount(c0, minlength=V)
    assert counts[p == 0].sum() == 0
    assert stats.chisquare(counts[p > 0], N * p[p > 0]).pvalue > 1e-4
    # the proposals follow the truncated drafter rows (here every proposal
    # row is row1): z_0 of each sequence
    sq = lex_topk(row1.astype(np.float64), kq)
    q = np.zeros(V)
    q[sq] = special.softmax(row1.astype(np.float64)[sq] / T)
    z = out["q_ids"][0, 0]
    assert list(z) == list(sq)
    np.testing.assert_allclose(out["q_probs"][0, 0], q[sq], rtol=1e-12)
    # next_draft[0] = z_a (a = commit_len): a draw from the truncated row1
    # wherever a proposal is left (a = 1)
    nd = out["next_draft"][:, 0]
    zc = np.bincount(nd[nd >= 0], minlength=V)
    N = int((nd >= 0).sum())
    assert N > 1000
    assert zc[q == 0].sum() == 0
    if kq > 1:
        assert stats.chisquare(zc[q > 0], N * q[q > 0]).pvalue > 1e-4


def test_lists_and_supports(orc):
    rng = np.random.default_rng(7)
    B, K, W, V, kp, kq = 16, 4, 5, 300, 8, 5
    logits = rng.normal(0, 2, (B, K + W, V)).astype(np.float32)
    prev_rows = rng.normal(0, 2, (B, W, V)).astype(np.float32)
    qi, qp = _prev_lists(prev_rows, 0.8, kq)
    off = rng.integers(0, 2, B).astype(np.int32)
    n = np.minimum(rng.integers(0, K, B), W - off).astype(np.int32)
    drafts = np.zeros((B, K - 1), np.int32)
    for b in range(B):
        for i in range(n[b]):
            drafts[b, i] = _draw(qi[b, off[b] + i], qp[b, off[b] + i], rng)
    out = orc.packed_topk_step(logits, K, W, kp, kq, drafts, n, qi, qp, off, 0.8, seed=1, it=4)
    np.testing.assert_allclose(out["q_probs"].sum(-1), 1.0, rtol=1e-12)
    for b in range(B):
        for j in range(W):
            assert list(out["q_ids"][b, j]) == list(lex_topk(logits[b, K + j].astype(np.float64), kq))
        a = out["commit_len"][b]
        for j in range(out["next_len"][b]):
            assert out["next_draft"][b, j] in out["q_ids"][b, a + j]
        h = out["accept_len"][b]
        c = out["committed"][b, h] if h < a else None
        if c is not None:  # the correction or bonus lies in the target's top kp
            assert c in lex_topk(logits[b, h].astype(np.float64), kp)


def test_draft_outside_its_list_is_rejected(orc):
    rng = np.random.default_rng(8)
    B, K, W, V, k = 1, 3, 3, 20, 4
    logits = rng.normal(0, 2, (B, K + W, V)).astype(np.float32)
    qi, qp = _prev_lists(rng.normal(0, 2, (B, W, V)).astype(np.float32), 1.0, k)
    bad = [v for v in range(V) if v not in qi[0, 0]][0]
    with pytest.raises(ValueError):
        orc.packed_topk_step(logits, K, W, k, k, np.array([[bad, 0]]), np.array([1]), qi, qp,
                             np.array([0]), 1.0)
