"""Pins of the oracle's SPOT verifier with the target's own position selection
([SPOT] App. A.1, Props. 1-2).

- Drafter invariance: on a toy block-diffusion target, the commitments of
  speculative rounds over arbitrary draft trees are the draft-free
  trajectory, token for token and position for position, at T = 0 and with
  the shared Gumbel table at T > 0 (the draft-free trajectory is the oracle's
  own answer for empty trees, one commitment per call).
- Position selection ranks masked positions by their largest probability,
  not their largest logit; ties go to the lowest position; unmasked positions
  never count.
- The accepted path is the longest chain of children that equal the target's
  transition of their parent's state (checked by enumerating root paths); a
  full block commits nothing more.
"""
import itertools

import numpy as np
import pytest

import oracle

MASK = -1


class ToyBlock:
    """Logits of a toy block-diffusion target: a seeded normal row for every
    (block state, position)."""

    def __init__(self, L, V, seed, scale=2.0):
        self.L, self.V, self.seed, self.scale = L, V, seed, scale

    def row(self, state, s):
        key = [self.seed, s] + [t + 1 for t in state]
        return np.random.default_rng(key).normal(0, self.scale, self.V).astype(np.float32)

    def rows(self, states):
        """[1, len(states), L, V] rows of every state."""
        out = np.zeros((1, len(states), self.L, self.V), np.float32)
        for i, st in enumerate(states):
            for s in range(self.L):
                if st[s] == MASK:
                    out[0, i, s] = self.row(st, s)
        return out


def mask_of(state):
    return sum(1 << s for s, t in enumerate(state) if t == MASK)


def commit(state, s, v):
    st = list(state)
    assert st[s] == MASK
    st[s] = v
    return tuple(st)


def draft_free(tgt, x0, T, seed, pos):
    """The draft-free trajectory: the oracle's commitment for an empty tree,
    one transition per call, until the block is full."""
    traj, x = [], x0
    while MASK in x:
        r = oracle.verify_spot(tgt.rows([x]), np.zeros((1, 0)), np.zeros((1, 0)),
                               np.zeros((1, 0)), [mask_of(x)], T=T, seed=seed, pos_base=[pos])
        assert r["path_len"][0] == 0 and r["commit_count"][0] == 1
        s, v = int(r["commit_pos"][0]), int(r["commit_tok"][0])
        traj.append((s, v))
        x = commit(x, s, v)
    return traj


def random_tree(x, orbit, k, rng, N, p_right=0.6, V=10):
    """A draft tree rooted at state x (= orbit state k): every node gets up to
    three children; a child repeats the orbit's next commitment with
    probability p_right when its parent lies on the orbit, else it commits a
    random token at a random masked position (duplicates allowed)."""
    parent, pos, tok, states, on = [], [], [], [x], [k]
    frontier = [-1]
    while frontier and len(parent) < N:
        y = frontier.pop(0)
        ys, yk = states[y + 1], on[y + 1]
        masked = [s for s in range(len(ys)) if ys[s] == MASK]
        if not masked:
            continue
        for _ in range(int(rng.integers(1, 4))):
            if len(parent) >= N:
                break
            if yk is not None and yk < len(orbit) and rng.random() < p_right:
                s, v = orbit[yk]
                nk = yk + 1
            else:
                s, v = int(rng.choice(masked)), int(rng.integers(V))
                nk = yk + 1 if (yk is not None and yk < len(orbit)
                                and (s, v) == orbit[yk]) else None
            parent.append(y)
            pos.append(s)
            tok.append(v)
            states.append(commit(ys, s, v))
            on.append(nk)
            frontier.append(len(parent) - 1)
    return parent, pos, tok, states


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_speculative_rounds_follow_the_draft_free_trajectory(orc, T, seed):
    L, V, pos = 7, 10, 1000 * seed
    tgt = ToyBlock(L, V, seed)
    x0 = (MASK,) * L
    orbit = draft_free(tgt, x0, T, seed, pos)
    assert len(orbit) == L
    rng = np.random.default_rng(seed)
    x, got, accepted = x0, [], 0
    while MASK in x:
        k = len(got)
        parent, npos, ntok, states = random_tree(x, orbit, k, rng, N=12)
        N = len(parent)
        r = orc.verify_spot(tgt.rows(states), np.array([parent]), np.array([npos]),
                            np.array([ntok]), [mask_of(x)], T=T, seed=seed, pos_base=[pos],
                            max_depth=max(N, 1))
        for d in range(int(r["path_len"][0])):
            n = int(r["path_nodes"][0, d])
            got.append((npos[n], ntok[n]))
            x = commit(x, npos[n], ntok[n])
        accepted += int(r["path_len"][0])
        if r["commit_pos"][0] >= 0:
            s, v = int(r["commit_pos"][0]), int(r["commit_tok"][0])
            got.append((s, v))
            x = commit(x, s, v)
        assert r["commit_count"][0] == r["path_len"][0] + (1 if r["commit_pos"][0] >= 0 else 0)
    assert got == orbit
    assert accepted > 0


def test_position_selection_uses_probabilities_and_lowest_ties(orc):
    L, V = 4, 64
    rows = np.full((1, 1, L, V), -10.0, np.float32)
    rows[0, 0, 0, :] = 4.9          # flat: largest logit 5 but a small largest probability
    rows[0, 0, 0, 3] = 5.0
    rows[0, 0, 1, 7] = 3.0          # one dominant token: largest probability near 1
    rows[0, 0, 3, 9] = 50.0         # not masked: never selected
    r = orc.verify_spot(rows, np.zeros((1, 0)), np.zeros((1, 0)), np.zeros((1, 0)), [0b0111])
    assert r["commit_pos"][0] == 1 and r["commit_tok"][0] == 7
    # position 2 gets the same row as position 1: an exact tie, the lower one wins
    rows[0, 0, 2] = rows[0, 0, 1]
    r = orc.verify_spot(rows, np.zeros((1, 0)), np.zeros((1, 0)), np.zeros((1, 0)), [0b0110])
    assert r["commit_pos"][0] == 1 and r["flags"][0] == 0
    r = orc.verify_spot(rows, np.zeros((1, 0)), np.zeros((1, 0)), np.zeros((1, 0)), [0b0100])
    assert r["commit_pos"][0] == 2


def test_path_is_the_longest_chain_of_target_transitions(orc):
    """Every root path is checked: the accepted path is the deepest chain in
    which each node commits its parent state's transition and is the lowest
    such child; no other chain of that kind is as deep."""
    L, V = 6, 8
    rng = np.random.default_rng(7)
    for trial in range(30):
        tgt = ToyBlock(L, V, 100 + trial)
        x0 = tuple(MASK if rng.random() < 0.8 else int(rng.integers(V)) for _ in range(L))
        if MASK not in x0:
            continue
        orbit = draft_free(tgt, x0, 0.0, 5, 0)
        parent, npos, ntok, states = random_tree(x0, orbit, 0, rng, N=10, p_right=0.7, V=V)
        N = len(parent)
        r = orc.verify_spot(tgt.rows(states), np.array([parent]), np.array([npos]),
                            np.array([ntok]), [mask_of(x0)], T=0.0, seed=5, max_depth=max(N, 1))
        sp, sv = r["state_pos"][0], r["state_tok"][0]

        def good(n):
            p = parent[n]
            if (npos[n], ntok[n]) != (sp[p + 1], sv[p + 1]):
                return False
            return all(not ((npos[m], ntok[m]) == (sp[p + 1], sv[p + 1]) and parent[m] == p)
                       for m in range(n))

        best = []
        for n in range(N):  # the chain ending at n, if all of it is good
            chain, m = [], n
            while m >= 0 and good(m):
                chain.append(m)
                m = parent[m]
            if m == -1 and len(chain) > len(best):
                best = chain[::-1]
        assert list(r["path_nodes"][0, :len(best)]) == best
        assert r["path_len"][0] == len(best)
        for n in range(N):
            assert r["match"][0, n] == int((npos[n], ntok[n]) == (sp[parent[n] + 1],
                                                                   sv[parent[n] + 1]))


def test_full_block_commits_nothing_more(orc):
    L, V = 3, 8
    tgt = ToyBlock(L, V, 9)
    x0 = (MASK,) * L
    orbit = draft_free(tgt, x0, 0.0, 1, 0)
    states = [x0]
    for s, v in orbit:
        states.append(commit(states[-1], s, v))
    parent = [-1, 0, 1]
    r = orc.verify_spot(tgt.rows(states), np.array([parent]), np.array([[s for s, _ in orbit]]),
                        np.array([[v for _, v in orbit]]), [mask_of(x0)])
    assert r["path_len"][0] == 3 and r["commit_count"][0] == 3 and r["commit_pos"][0] == -1
    assert r["state_pos"][0, 3] == -1


def test_commitment_must_be_at_a_masked_position(orc):
    rows = np.zeros((1, 2, 2, 8), np.float32)
    with pytest.raises(ValueError):
        orc.verify_spot(rows, np.array([[-1]]), np.array([[1]]), np.array([[0]]), [0b01])
