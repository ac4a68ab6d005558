"""Pins of the oracle's any-order Packed-SS iteration ([PackedSS] App. C,
Alg. 3, Prop. C.1; confidence scores of App. E.6).

- Prop. C.1 (greedy correctness under the chosen orders): a whole decode by
  Alg. 3 on a toy any-order target, with the oracle doing each iteration's
  verify step and the confidence order of App. E.6, returns what a serial
  reference returns when it generates each iteration's A_t tokens greedily,
  one at a time, in the same order and with the same end rule.
- The left-to-right order on a full draft reduces to the greedy Packed-SS
  step of Alg. 1.
- A small worked case: the rank order, the verifier's token at the first
  mismatch, the retained drafts and their confidence order, and an
  accepted EOS that cuts the pairs beyond it.
"""
import numpy as np
import pytest
from scipy import special

import oracle

EOS = 3


class ToyAnyOrder:
    """An any-order target and its drafter: the logits at position j given a
    set of known (position, token) pairs come from a seeded hash; the
    drafter's are the target's plus noise."""

    def __init__(self, V, seed, noise=0.6):
        self.V, self.seed, self.noise = V, seed, noise

    def _key(self, ctx, j):
        return [self.seed, j] + [x for pt in sorted(ctx) for x in pt]

    def target(self, ctx, j):
        return np.random.default_rng(self._key(ctx, j)).normal(0, 2, self.V).astype(np.float32)

    def drafter(self, ctx, j):
        k = self._key(ctx, j) + [7777]
        return (self.target(ctx, j) +
                np.random.default_rng(k).normal(0, self.noise, self.V)).astype(np.float32)


def alg3(tgt, Lmax, W, eos):
    """Alg. 3 with the oracle's iteration; returns the output (position ->
    token, up to E) and each iteration's (order positions, A_t, E before)."""
    P = {}            # accepted position -> token
    D = {}            # position -> draft token
    score = {}        # position -> confidence of its draft
    E, trace = Lmax, []
    while any(j not in P for j in range(1, E + 1)):
        ell = min(j for j in range(1, E + 1) if j not in P)
        U = [j for j in range(ell, min(E, ell + W - 1) + 1) if j not in P]
        u = len(U)
        with_d = sorted((j for j in U if j in D), key=lambda j: (-score[j], j))
        pi = with_d + [j for j in U if j not in D]     # App. E.6
        kappa = 0
        while kappa < u and pi[kappa] in D:
            kappa += 1
        nreq = min(kappa + 1, u)
        ctx = set(P.items())
        rows = np.zeros((1, W + W, tgt.V), np.float32)
        for r in range(nreq):
            rows[0, r] = tgt.target(ctx | {(pi[s], D[pi[s]]) for s in range(r)}, pi[r])
        for i, j in enumerate(U):
            rows[0, W + i] = tgt.drafter(ctx, j)
        wp = np.full((1, W), -1, np.int32)
        wp[0, :u] = U
        od = np.full((1, W), -1, np.int32)
        od[0, :u] = [U.index(j) for j in pi]
        dr = np.full((1, W), -1, np.int32)
        dr[0, :u] = [D.get(j, -1) for j in U]
        out = oracle.packed_anyorder_step(rows, W, W, [u], wp, od, dr, [E], eos_id=eos)
        A = min(int(out["accept_len"][0]) + 1, u)
        trace.append((pi, A, E))
        for k in range(int(out["commit_len"][0])):
            P[int(out["commit_pos"][0, k])] = int(out["commit_tok"][0, k])
        E = int(out["end_pos"][0])
        P = {j: v for j, v in P.items() if j <= E}
        D, score = {}, {}
        for i in range(u):
            if out["next_draft"][0, i] >= 0:
                D[U[i]] = int(out["next_draft"][0, i])
                score[U[i]] = float(out["score"][0, i])
        # the order output is the same ranking of the retained positions
        ranked = [U[i] for i in out["next_order"][0] if i >= 0]
        assert ranked == sorted(D, key=lambda j: (-score[j], j))
    return [P[j] for j in range(1, E + 1)], trace


def serial_reference(tgt, trace, eos):
    """Prop. C.1's serial reference: each iteration generates A_t tokens
    greedily at pi_t(1..A_t), each conditioned on its own accepted pairs and
    the tokens generated before it in the group."""
    P, E = {}, trace[0][2]
    for pi, A, _ in trace:
        ctx = set(P.items())
        group = []
        for r in range(A):
            y = int(np.argmax(tgt.target(ctx | set(group), pi[r])))
            group.append((pi[r], y))
        for j, y in group:
            if y == eos and j < E:
                E = j
        for j, y in group:
            if j <= E:
                P[j] = y
        P = {j: v for j, v in P.items() if j <= E}
    return [P[j] for j in range(1, E + 1)]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("W", [1, 3, 6])
def test_greedy_correctness_under_confidence_orders(orc, seed, W):
    tgt = ToyAnyOrder(V=8, seed=seed, noise=0.5 if seed % 2 else 1.5)
    out, trace = alg3(tgt, Lmax=14, W=W, eos=EOS)
    assert out == serial_reference(tgt, trace, EOS)


def test_greedy_correctness_without_eos(orc):
    """Long decodes (no EOS) in which drafts are accepted and the confidence
    orders differ from the textual order."""
    multi = reordered = 0
    for seed in range(8):
        tgt = ToyAnyOrder(V=6, seed=100 + seed, noise=0.4)
        out, trace = alg3(tgt, Lmax=24, W=5, eos=-1)
        assert out == serial_reference(tgt, trace, -1) and len(out) == 24
        multi += sum(A > 1 for _, A, _ in trace)
        reordered += sum(pi != sorted(pi) for pi, _, _ in trace)
    assert multi > 5 and reordered > 5


def test_left_to_right_order_is_the_packed_step(orc):
    """Identity order, drafts at the first W - 1 positions: the same h, A and
    committed tokens as the Alg. 1 greedy step on the same rows."""
    rng = np.random.default_rng(3)
    B, W, V = 20, 5, 16
    K = W
    rows = rng.normal(0, 2, (B, K + W, V)).astype(np.float32)
    vt = rows[:, :K].argmax(-1)
    drafts = np.where(rng.random((B, K - 1)) < 0.7, vt[:, :K - 1], (vt[:, :K - 1] + 1) % V)
    n = np.full(B, K - 1, np.int32)
    ref = orc.packed_step(rows, K, W, drafts, n, T=0.0)
    wp = np.tile(np.arange(1, W + 1, dtype=np.int32), (B, 1))
    od = np.tile(np.arange(W, dtype=np.int32), (B, 1))
    dr = np.concatenate([drafts, -np.ones((B, 1), np.int64)], 1)
    out = orc.packed_anyorder_step(rows, K, W, np.full(B, W), wp, od, dr, np.full(B, 100))
    assert np.array_equal(out["accept_len"], ref["accept_len"])
    assert np.array_equal(out["commit_len"], ref["commit_len"])
    for b in range(B):
        a = ref["commit_len"][b]
        assert list(out["commit_tok"][b, :a]) == list(ref["committed"][b, :a])
        assert list(out["commit_pos"][b, :a]) == list(range(1, a + 1))


def test_worked_case(orc):
    """Window positions 5..8, ranks over indices (2, 0, 3, 1), drafts at 5, 7
    and 8: rank 0 (position 7) matches, rank 1 (position 5) does not; A = 2
    commits (7, d7) and (5, v).  Retained: positions 6 and 8, ordered by
    their proposal probabilities."""
    V, W = 10, 4
    rows = np.full((1, W + W, V), -5.0, np.float32)
    rows[0, 0, 4] = 5.0   # rank 0: verifier says 4 at position 7
    rows[0, 1, 6] = 5.0   # rank 1: verifier says 6 at position 5 (draft was 2)
    for i, (z, top) in enumerate([(1, 1.0), (2, 3.0), (0, 2.0), (9, 6.0)]):
        rows[0, W + i, z] = top  # proposals at positions 5, 6, 7, 8
    wp = np.array([[5, 6, 7, 8]])
    od = np.array([[2, 0, 3, 1]])
    dr = np.array([[2, -1, 4, 7]])
    out = orc.packed_anyorder_step(rows, W, W, [4], wp, od, dr, [30])
    assert out["accept_len"][0] == 1 and out["commit_len"][0] == 2
    assert list(out["commit_pos"][0, :2]) == [7, 5] and list(out["commit_tok"][0, :2]) == [4, 6]
    assert list(out["next_draft"][0]) == [-1, 2, -1, 9]
    s = out["score"][0]
    assert abs(s[3] - special.softmax(rows[0, W + 3].astype(np.float64))[9]) < 1e-12
    assert list(out["next_order"][0]) == [3, 1, -1, -1]   # position 8 scores higher than 6
    # the verifier's token at rank 0 is EOS: position 7 becomes the end, so
    # the pair at rank 1 survives only because 5 <= 7, and position 8 is
    # no longer retained
    out = orc.packed_anyorder_step(rows, W, W, [4], wp, od, dr, [30], eos_id=4)
    assert out["end_pos"][0] == 7 and out["commit_len"][0] == 2
    assert list(out["next_draft"][0]) == [-1, 2, -1, -1]
