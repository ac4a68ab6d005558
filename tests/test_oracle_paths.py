"""Pins of the oracle's four full procedures (greedy, sample, tree, packed)
against what the pages fix: plain argmax decoding, the Packed-SS worked
example, the stopping rule, the pathwise-dominance and distributional
theorems, the acceptance-equals-1-TV check, the expected accepted length, and
the tree verifier's path structure and drafter invariance."""
import itertools
import math
import os

import numpy as np
import pytest
from scipy import special, stats

from datagen import random_trees

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


class ToyAR:
    def __init__(self, V, seed, scale=2.0):
        self.V, self.seed, self.scale = V, seed, scale
        self._c = {}

    def logits(self, prefix):
        prefix = tuple(int(t) for t in prefix)
        if prefix not in self._c:
            rng = np.random.default_rng([self.seed, len(prefix)] + [t + 7 for t in prefix])
            self._c[prefix] = rng.normal(0, self.scale, self.V).astype(np.float32)
        return self._c[prefix]


# --------------------------------------------------------------------------- greedy

def test_greedy_loop_equals_argmax_decoding(orc):
    # [PackedSS] App. B.2 "Greedy decoding" / [SPOT] Prop. 1: greedy verification
    # reproduces plain argmax decoding token for token, whatever the drafts.
    V, K, L = 50, 5, 60
    tgt = ToyAR(V, seed=41)
    ref = []
    while len(ref) < L:
        ref.append(int(np.argmax(tgt.logits(ref))))
    rng = np.random.default_rng(0)
    out, calls = [], 0
    while len(out) < L:
        draft = []
        for i in range(K):
            good = int(np.argmax(tgt.logits(out + draft)))
            draft.append(good if rng.random() < 0.7 else int(rng.integers(V)))
        rows = np.stack([tgt.logits(out + draft[:i]) for i in range(K + 1)])[None]
        r = orc.verify_greedy(rows, np.array([draft]))
        h = int(r["accept_len"][0])
        assert draft[:h] == ref[len(out):len(out) + h]
        out += draft[:h] + [int(r["next_token"][0])]
        calls += 1
    assert out[:L] == ref
    assert calls < L  # some drafts were accepted


def test_greedy_ragged_and_ties(orc):
    V = 8
    rows = np.zeros((3, 4, V), np.float32)
    rows[:, :, 2] = 1.0
    rows[:, :, 5] = 1.0          # exact tie: the lower id (2) is the argmax
    ids = np.array([[2, 2, 2], [2, 5, 2], [5, 2, 2]])
    r = orc.verify_greedy(rows, ids, draft_len=np.array([3, 1, 0]))
    assert list(r["accept_len"]) == [3, 1, 0]
    assert list(r["next_token"]) == [2, 2, 2]


# --------------------------------------------------------------------------- packed

def _fig2():
    d = {}
    for line in open(os.path.join(GOLDEN, "packed_fig2.txt")):
        line = line.split("#")[0].split()
        if line:
            d[line[0]] = line[1:]
    return d


def test_packed_fig2_worked_example(orc):
    g = _fig2()
    W = int(g["W"][0])
    K = W
    tok = {"d1": 3, "d2": 4, "d3": 5, "v2": 7, "z1": 1, "z2": 2, "z3": 8, "z4": 9}
    V = 16
    logits = np.zeros((1, K + W, V), np.float32)
    for i, t in enumerate([tok["d1"], tok["v2"], 11, 12]):   # verifier rows
        logits[0, i, t] = 5.0
    for j in range(W):                                        # proposal rows
        logits[0, K + j, tok["z%d" % (j + 1)]] = 5.0
    prev = [tok[s] for s in g["prev_draft"]]
    r = orc.packed_step(logits, K, W, np.array([prev]), np.array([len(prev)]))
    assert r["accept_len"][0] == int(g["h"][0])
    assert r["commit_len"][0] == int(g["A"][0])
    assert list(r["committed"][0, :2]) == [tok[s] for s in g["committed"]]
    nl = int(r["next_len"][0])
    assert list(r["next_draft"][0, :nl]) == [tok[s] for s in g["next_draft"]]
    assert np.all(r["next_draft"][0, nl:] == -1)
    # greedy drafts carry q = 1; confidence is the max softmax of each row
    assert np.allclose(r["next_q_at_draft"][0, :nl], 1.0)
    conf = special.softmax(logits[0, K:].astype(np.float64), axis=-1).max(-1)
    assert np.allclose(r["confidence"][0], conf, rtol=1e-12)


def _onehot_rows(tokens, V, hi=5.0):
    rows = np.zeros((len(tokens), V), np.float32)
    for i, t in enumerate(tokens):
        rows[i, t] = hi
    return rows


def test_packed_stopping_index(orc):
    # [PackedSS] Alg. 1 line 7: a = min({A, L+|P|-|P_{t-1}|} ∪ {i : C_i = EOS})
    V, K, W, EOS = 10, 4, 4, 9
    z = [1, 2, 3, 4]
    def run(verify_argmax, prev, eos=-1, rem=None):
        lg = np.concatenate([_onehot_rows(verify_argmax, V), _onehot_rows(z, V)])[None]
        return orc.packed_step(lg, K, W, np.array([prev + [0] * (K - 1 - len(prev))]),
                               np.array([len(prev)]), eos_id=eos,
                               remaining=None if rem is None else np.array([rem]))
    r = run([5, 6, 7, 8], [5, 6, 7])                 # all accepted, bonus 8: A = 4
    assert (r["accept_len"][0], r["commit_len"][0]) == (3, 4)
    assert r["next_len"][0] == 0
    r = run([5, EOS, 7, 8], [5, EOS, 7], eos=EOS)    # accepted EOS at C_2 stops there
    assert (r["accept_len"][0], r["commit_len"][0]) == (3, 2)
    assert list(r["committed"][0]) == [5, EOS, -1, -1]
    assert list(r["next_draft"][0, :2]) == [3, 4]
    r = run([5, 6, 7, 8], [5, 6, 7], rem=2)          # length cap
    assert r["commit_len"][0] == 2
    r = run([EOS, 6, 7, 8], [5, 6, 7], eos=EOS)      # correction is EOS
    assert (r["accept_len"][0], r["commit_len"][0]) == (0, 1)
    assert list(r["committed"][0, :1]) == [EOS]
    r = run([5, 6, 7, 8], [])                        # D_0 is empty: one AR token
    assert (r["accept_len"][0], r["commit_len"][0]) == (0, 1)
    assert list(r["committed"][0, :1]) == [5]
    assert list(r["next_draft"][0, :3]) == [2, 3, 4]


def _monotone_drafter(x_true, V, rng):
    """Assumption 3.1: position k (1-indexed) is predicted correctly from c
    verified tokens iff c >= c*_k, for thresholds c*_k <= k."""
    cstar = [int(rng.integers(0, k + 1)) for k in range(1, len(x_true) + 1)]
    def draft(k, c):
        if k > len(x_true):
            return 0
        return x_true[k - 1] if c >= cstar[k - 1] else (x_true[k - 1] + 1) % V
    return draft


@pytest.mark.parametrize("seed", range(6))
def test_packed_greedy_dominates_linear(orc, seed):
    # [PackedSS] Thm 3.2: under Assumption 3.1, Packed-SS needs no more model
    # calls than Linear-SS for any output length; both equal greedy AR output.
    V, W, L = 12, 5, 40
    K = W
    tgt = ToyAR(V, seed=100 + seed)
    x = []
    while len(x) < L + W + 2:
        x.append(int(np.argmax(tgt.logits(x))))
    dr = _monotone_drafter(x, V, np.random.default_rng(seed))

    P, D, nfe = [], [], 0
    packed_nfe = {}
    while len(P) < L:
        rows = [tgt.logits(P + D[:i]) if i <= len(D) else np.zeros(V, np.float32)
                for i in range(K)]
        c = len(P)
        rows += list(_onehot_rows([dr(c + j + 1, c) for j in range(W)], V))
        r = orc.packed_step(np.stack(rows)[None], K, W,
                            np.array([D + [0] * (K - 1 - len(D))]), np.array([len(D)]))
        nfe += 1
        a = int(r["commit_len"][0])
        P += list(r["committed"][0, :a])
        D = list(r["next_draft"][0, :int(r["next_len"][0])])
        for ell in range(1, len(P) + 1):
            packed_nfe.setdefault(ell, nfe)
    assert P[:L] == x[:L]

    P, nfe = [], 0
    linear_nfe = {}
    while len(P) < L:
        c = len(P)
        d = [dr(c + j + 1, c) for j in range(W)]
        nfe += 1                                    # drafting call
        rows = np.stack([tgt.logits(P + d[:i]) for i in range(W + 1)])[None]
        r = orc.verify_greedy(rows, np.array([d]))
        nfe += 1                                    # verification call
        h = int(r["accept_len"][0])
        P += d[:h] + [int(r["next_token"][0])]
        for ell in range(1, len(P) + 1):
            linear_nfe.setdefault(ell, nfe)
    assert P[:L] == x[:L]
    for ell in range(1, L + 1):
        assert packed_nfe[ell] <= linear_nfe[ell]


def test_packed_sampling_preserves_target_law(orc):
    # [PackedSS] Thm 3.3: at T = 1 the first L tokens produced by the Packed-SS
    # loop (stored proposals, residual from the stored Q row, drafts keyed by
    # the call index) follow the target's chain rule.
    V, W, L, B, T = 3, 3, 3, 30000, 1.0
    K = W
    tgt = ToyAR(V, seed=7, scale=1.2)
    dft = ToyAR(V, seed=8, scale=1.2)
    P = [[] for _ in range(B)]
    D = [[] for _ in range(B)]
    Dq = [[] for _ in range(B)]
    prev_rows = np.zeros((B, W, V), np.float32)
    a_prev = np.zeros(B, np.int32)
    it = 0
    while any(len(p) < L for p in P):
        it += 1
        lg = np.zeros((B, K + W, V), np.float32)
        for b in range(B):
            for i in range(len(D[b]) + 1):
                lg[b, i] = tgt.logits(P[b] + D[b][:i])
            for j in range(W):
                lg[b, K + j] = dft.logits(P[b] + [V + j])
        pd = np.zeros((B, K - 1), np.int32)
        pq = np.ones((B, K - 1), np.float32)
        for b in range(B):
            pd[b, :len(D[b])] = D[b]
            pq[b, :len(D[b])] = Dq[b]
        rem = np.array([max(L - len(p), 1) for p in P])
        r = orc.packed_step(lg, K, W, pd, np.array([len(d) for d in D]), pq, prev_rows,
                            a_prev, T=T, seed=2024, it=it,
                            pos_base=np.array([len(p) for p in P]), remaining=rem)
        for b in range(B):
            if len(P[b]) >= L:
                continue
            a = int(r["commit_len"][b])
            P[b] += [int(t) for t in r["committed"][b, :a]]
            nl = int(r["next_len"][b])
            D[b] = [int(t) for t in r["next_draft"][b, :nl]]
            Dq[b] = [float(q) for q in r["next_q_at_draft"][b, :nl]]
        prev_rows = lg[:, K:].copy()
        a_prev = r["commit_len"].copy()
    counts = np.zeros((V,) * L)
    for p in P:
        counts[tuple(p[:L])] += 1
    law = np.zeros((V,) * L)
    for s in itertools.product(range(V), repeat=L):
        law[s] = np.prod([special.softmax(tgt.logits(list(s[:j])).astype(np.float64) / T)[s[j]]
                          for j in range(L)])
    assert stats.chisquare(counts.ravel(), B * law.ravel()).pvalue > 1e-4


# --------------------------------------------------------------------------- sample

def test_sample_acceptance_matches_tv(orc):
    # [SPOT] App. B.4: the empirical acceptance rate of the RS verifier is within
    # 0.002 of 1 - D_TV; the emitted token follows p (chi-square).
    V, B = 6, 2_000_000
    rng = np.random.default_rng(9)
    x = rng.normal(0, 1.5, V).astype(np.float32)
    y = (x + rng.normal(0, 1.0, V)).astype(np.float32)
    p = special.softmax(x.astype(np.float64))
    q = special.softmax(y.astype(np.float64))
    tgt = np.broadcast_to(x, (B, 2, V))
    drf = np.broadcast_to(y, (B, 1, V))
    ids = rng.choice(V, size=(B, 1), p=q)
    r = orc.verify_sample(tgt, drf, ids, seed=17, want_tv=True)
    acc = r["accept_len"].mean()
    tvd = 0.5 * np.abs(p - q).sum()
    assert abs(acc - (1 - tvd)) < 0.002
    assert r["tv"][0, 0] == pytest.approx(tvd, abs=1e-7)
    first = np.where(r["accept_len"] == 1, ids[:, 0], r["next_token"])
    counts = np.bincount(first, minlength=V)
    assert stats.chisquare(counts, B * p).pvalue > 1e-4


def test_sample_expected_emitted_length(orc):
    # [TwoTrade] App. C Prop. 1: with independent per-position acceptance of mean
    # mu, the expected number of emitted tokens is sum_{n=0}^{K} mu^n.
    V, K, B = 8, 6, 200_000
    rng = np.random.default_rng(10)
    x = rng.normal(0, 1.5, V).astype(np.float32)
    y = (x + rng.normal(0, 0.8, V)).astype(np.float32)
    p = special.softmax(x.astype(np.float64))
    q = special.softmax(y.astype(np.float64))
    mu = 1 - 0.5 * np.abs(p - q).sum()
    r = orc.verify_sample(np.broadcast_to(x, (B, K + 1, V)), np.broadcast_to(y, (B, K, V)),
                          rng.choice(V, size=(B, K), p=q), seed=3, want_tv=False)
    emitted = r["accept_len"] + 1
    expect = sum(mu ** n for n in range(K + 1))
    assert abs(emitted.mean() - expect) < 4 * emitted.std() / math.sqrt(B)


def test_sample_lenient_reductions(orc):
    # lam = 1 (ratio) and mu = 0 (linear) give bit-identical outputs to lossless
    rng = np.random.default_rng(11)
    B, K, V = 64, 5, 40
    x = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    y = (x[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    ids = rng.integers(0, V, (B, K))
    base = orc.verify_sample(x, y, ids, seed=5)
    for mode, lam in ((1, 1.0), (2, 0.0)):
        r = orc.verify_sample(x, y, ids, seed=5, mode=mode, lam=lam)
        for k in base:
            assert np.array_equal(base[k], r[k], equal_nan=True), k
    # leniency never lowers the accepted length on the same random numbers
    for lam in (2.0, 4.0, 8.0):
        r = orc.verify_sample(x, y, ids, seed=5, mode=1, lam=lam)
        assert np.all(r["accept_len"] >= base["accept_len"])


def test_sample_per_row_outputs(orc):
    rng = np.random.default_rng(12)
    B, K, V = 3, 4, 30
    Tp, Tq = float(np.float32(0.7)), float(np.float32(1.3))  # temperatures are fp32 in the ABI
    x = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    y = rng.normal(0, 2, (B, K, V)).astype(np.float32)
    ids = rng.integers(0, V, (B, K))
    dl = np.array([4, 2, 0])
    r = orc.verify_sample(x, y, ids, draft_len=dl, T_p=Tp, T_q=Tq, seed=1)
    for b in range(B):
        for i in range(K + 1):
            if i <= dl[b]:
                assert r["lse_p"][b, i] == pytest.approx(
                    special.logsumexp(x[b, i].astype(np.float64) / Tp), rel=1e-14)
            else:
                assert np.isnan(r["lse_p"][b, i])
        for i in range(K):
            if i < dl[b]:
                p = special.softmax(x[b, i].astype(np.float64) / Tp)
                q = special.softmax(y[b, i].astype(np.float64) / Tq)
                assert r["p_at_draft"][b, i] == pytest.approx(p[ids[b, i]], rel=1e-13)
                assert r["q_at_draft"][b, i] == pytest.approx(q[ids[b, i]], rel=1e-13)
                assert r["tv"][b, i] == pytest.approx(0.5 * np.abs(p - q).sum(), abs=1e-14)
            else:
                assert np.isnan(r["tv"][b, i])
    assert r["accept_len"][2] == 0


# --------------------------------------------------------------------------- tree

@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tree_path_is_deepest_matching_root_path(orc, T):
    # [SPOT] App. A.1 "State-equality verifier": a node is accepted only if its
    # whole root path matches; the result is the deepest such path.  Checked by
    # enumerating all root paths.
    B, N, V = 40, 16, 4
    parent, pos, depth = random_trees(B, N, L=8, max_depth=5, max_children=3, seed=5)
    rng = np.random.default_rng(13)
    lg = rng.normal(0, 1, (B, N, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, N))
    r = orc.verify_tree(lg, parent, pos, tok, T=T, seed=9, max_depth=6)
    for b in range(B):
        m = r["match"][b].astype(bool)
        if T == 0.0:
            assert np.array_equal(m, lg[b].argmax(-1) == tok[b])
        best, bestd = -1, 0
        for n in range(N):
            path = [n]
            while parent[b, path[-1]] >= 0:
                path.append(parent[b, path[-1]])
            if all(m[k] for k in path) and len(path) > bestd:
                best, bestd = n, len(path)
        assert r["path_len"][b] == bestd
        assert r["commit_count"][b] == bestd + 1
        nodes = []
        n = best
        while n >= 0:
            nodes.append(n)
            n = parent[b, n]
        nodes = nodes[::-1] + [-1] * (6 - len(nodes))
        assert list(r["path_nodes"][b]) == nodes[:6]


class ToyBlock:
    """A toy block-diffusion target over L positions: logits for every
    (state, position) from a seeded hash; position selection s*(x) picks the
    masked position with the largest maximum probability ([SPOT] §4.1)."""

    MASK = -1

    def __init__(self, L, V, seed):
        self.L, self.V, self.seed = L, V, seed
        self._c = {}

    def logits(self, x, s):
        k = (tuple(x), s)
        if k not in self._c:
            rng = np.random.default_rng([self.seed, s] + [t + 2 for t in x])
            self._c[k] = rng.normal(0, 1.5, self.V).astype(np.float32)
        return self._c[k]

    def s_star(self, x):
        masked = [s for s in range(self.L) if x[s] == self.MASK]
        conf = [special.softmax(self.logits(x, s).astype(np.float64)).max() for s in masked]
        return masked[int(np.argmax(conf))]


@pytest.mark.parametrize("T,seed", [(0.0, 1), (1.0, 2), (1.0, 3), (0.7, 4)])
def test_tree_drafter_invariance(orc, T, seed):
    # [SPOT] Props. 1-2 and App. A.3 Step 2: with the shared Gumbel table the
    # committed trajectory is the draft-free orbit of Phi_G, whatever tree the
    # drafter proposes.
    L, V, b = 6, 5, 3
    tb = ToyBlock(L, V, seed)
    def phi(x):
        s = tb.s_star(x)
        lg = tb.logits(x, s).astype(np.float64)
        if T == 0.0:
            v = orc.argmax(lg)
        else:
            v = orc.gumbel_argmax(lg / T, orc.key(seed, orc.ST_TREE, b, s, 0))[0]
        y = list(x)
        y[s] = v
        return y, s, v
    x = [ToyBlock.MASK] * L
    orbit = [x]
    while ToyBlock.MASK in x:
        x = phi(x)[0]
        orbit.append(x)
    rng = np.random.default_rng(seed)
    for trial in range(5):
        state, traj = [ToyBlock.MASK] * L, [[ToyBlock.MASK] * L]
        while ToyBlock.MASK in state:
            # drafter: a random tree whose nodes commit at s*(parent state),
            # with the right token only sometimes
            nodes = []     # (parent, pos, tok, state_after)
            for n in range(int(rng.integers(1, 9))):
                cands = [-1] + [k for k, nd in enumerate(nodes) if ToyBlock.MASK in nd[3]]
                par = cands[int(rng.integers(len(cands)))]
                ps = state if par < 0 else nodes[par][3]
                if ToyBlock.MASK not in ps:
                    continue
                y, s, v = phi(ps)
                if rng.random() < 0.4:
                    v = int(rng.integers(V))
                    y = list(ps)
                    y[s] = v
                nodes.append((par, s, v, y))
            N = len(nodes)
            lg = np.stack([tb.logits(state if p < 0 else nodes[p][3], s)
                           for p, s, _, _ in nodes])[None]
            # verify_tree keys the noise by (sequence, position): use sequence b
            r = orc.verify_tree(np.repeat(lg, b + 1, 0),
                                np.repeat([[nd[0] for nd in nodes]], b + 1, 0),
                                np.repeat([[nd[1] for nd in nodes]], b + 1, 0),
                                np.repeat([[nd[2] for nd in nodes]], b + 1, 0), T=T,
                                seed=seed, max_depth=N)
            plen = int(r["path_len"][b])
            for k in range(plen):
                state = nodes[int(r["path_nodes"][b, k])][3]
                traj.append(state)
            if ToyBlock.MASK in state:
                state = phi(state)[0]       # the verifier's own commitment
                traj.append(state)
        assert traj == orbit
