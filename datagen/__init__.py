"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds none of the verification arithmetic.  It builds logit rows
with the shapes and value distributions of the five workloads (i.i.d.
N(0, 2^2) logits, drafter = target + N(0, sigma^2), random draft trees,
Packed-SS state) and draws the drafter's own proposals with torch's generator.
The verify side's random numbers (acceptance uniforms, Gumbel noise) are not
made here: both implementations derive them from the counter hash.

All tensors are created on ``device`` with a ``torch.Generator`` seeded by
``seed``; bf16 rows are rounded from fp32 to nearest-even by torch.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

# The five workloads: sizes, dtypes and seeds of the verify problems.
CONFIGS = {
    "greedy_tiny": dict(kind="greedy", B=1, K=8, V=32000, dtype="f32", seed=0),
    "lossless_t1": dict(kind="sample", B=64, K=16, V=128256, dtype="bf16", seed=1,
                        sigma=0.5, T=1.0),
    "lenient_sweep": dict(kind="sample", B=128, K=16, V=151936, dtype="bf16", seed=2,
                          sigma=(0.25, 1.0), T=(0.7, 1.0), lam=(1.0, 2.0, 4.0, 8.0)),
    "tree": dict(kind="tree", B=32, N=64, V=151936, dtype="bf16", seed=3, L=32,
                 max_depth=8, max_children=4, T=(0.0, 1.0)),
    "packed": dict(kind="packed", B=256, K=32, W=32, V=151936, dtype="bf16", seed=4,
                   T=(0.0, 1.0)),
    # Packed-SS at T = 1 with top-k truncated target and drafter
    # distributions, k = 20 of 151,936 (the top-k the truncation passage
    # quotes for that vocabulary)
    "packed_topk": dict(kind="packed_topk", B=256, K=32, W=32, V=151936, dtype="bf16", seed=7,
                        kp=20, kq=20, T=1.0),
    # any-order Packed-SS steps: windows of 32 unresolved positions checked
    # in a random rank order, drafts at 90% of them
    "anyorder": dict(kind="anyorder", B=256, K=32, W=32, V=151936, dtype="bf16", seed=6),
    # SPOT trees with the target's own position selection: 32 trees of 8
    # drafted states over a 32-position block that starts fully masked
    "spot": dict(kind="spot", B=32, N=8, L=32, V=151936, dtype="bf16", seed=5,
                 max_depth=8, max_children=4, T=(0.0, 1.0)),
}

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _pick_tokens(rows: torch.Tensor, p_match: float, g, device) -> torch.Tensor:
    """Per row: the row's largest entry with probability p_match, else a uniform
    other id (the draft-quality recipe of the greedy workloads)."""
    V = rows.shape[-1]
    best = rows.float().argmax(dim=-1)
    other = torch.randint(0, V - 1, best.shape, generator=g, device=device)
    other = other + (other >= best).to(other.dtype)
    keep = torch.rand(best.shape, generator=g, device=device) < p_match
    return torch.where(keep, best, other).to(torch.int32)


def _draw_from_logits(rows: torch.Tensor, T: float, g, device) -> torch.Tensor:
    """The drafter's own proposal: one categorical draw per row from
    softmax(rows / T), by torch.multinomial (rows are flattened to 2-D)."""
    flat = rows.reshape(-1, rows.shape[-1]).float()
    probs = torch.softmax(flat / T, dim=-1)
    out = torch.multinomial(probs, 1, generator=g).reshape(rows.shape[:-1])
    return out.to(torch.int32)


@dataclasses.dataclass
class GreedyInputs:
    target: torch.Tensor      # [B, K+1, V]
    draft_ids: torch.Tensor   # [B, K] int32
    draft_len: torch.Tensor   # [B] int32


def greedy_inputs(B, K, V, dtype="f32", seed=0, p_match=0.8, device="cpu",
                  ragged=False) -> GreedyInputs:
    g = _gen(seed, device)
    target = _normal((B, K + 1, V), 2.0, g, device).to(_TORCH_DTYPE[dtype])
    ids = _pick_tokens(target[:, :K], p_match, g, device) if K > 0 else \
        torch.zeros((B, 0), dtype=torch.int32, device=device)
    if ragged:
        dl = torch.randint(0, K + 1, (B,), generator=g, device=device).to(torch.int32)
    else:
        dl = torch.full((B,), K, dtype=torch.int32, device=device)
    return GreedyInputs(target, ids, dl)


@dataclasses.dataclass
class SampleInputs:
    target: torch.Tensor      # [B, K+1, V]
    draft: torch.Tensor       # [B, K, V]
    draft_ids: torch.Tensor   # [B, K] int32, drawn from softmax(draft / T_q)
    draft_len: torch.Tensor   # [B] int32


def sample_inputs(B, K, V, dtype="bf16", seed=1, sigma=0.5, T=1.0, device="cpu",
                  ragged=False, target_std=2.0) -> SampleInputs:
    g = _gen(seed, device)
    tgt32 = _normal((B, K + 1, V), target_std, g, device)
    drf32 = tgt32[:, :K] + _normal((B, K, V), sigma, g, device)
    target = tgt32.to(_TORCH_DTYPE[dtype])
    draft = drf32.to(_TORCH_DTYPE[dtype])
    del tgt32, drf32
    if K > 0:
        ids = _draw_from_logits(draft, T, g, device)
    else:
        ids = torch.zeros((B, 0), dtype=torch.int32, device=device)
    if ragged:
        dl = torch.randint(0, K + 1, (B,), generator=g, device=device).to(torch.int32)
    else:
        dl = torch.full((B,), K, dtype=torch.int32, device=device)
    return SampleInputs(target, draft, ids, dl)


@dataclasses.dataclass
class TreeInputs:
    node_logits: torch.Tensor  # [B, N, V]
    parent: torch.Tensor       # [B, N] int32, -1 = child of the root
    node_pos: torch.Tensor     # [B, N] int32 in [0, L)
    node_tok: torch.Tensor     # [B, N] int32
    depth: np.ndarray          # [B, N] host-side depths (1 = child of root)


def random_trees(B, N, L=32, max_depth=8, max_children=4, seed=3):
    """Parents, positions and depths of B random draft trees (host numpy).
    Node n picks a uniform parent among the root and the earlier nodes that
    are shallower than max_depth and have fewer than max_children children;
    its block position is uniform among those not used on its root path."""
    rng = np.random.default_rng(seed)
    parent = np.full((B, N), -1, np.int32)
    pos = np.zeros((B, N), np.int32)
    depth = np.zeros((B, N), np.int32)
    for b in range(B):
        children = np.zeros(N + 1, np.int64)  # index N is the root
        for n in range(N):
            cand = [N] if children[N] < max_children else []
            cand += [m for m in range(n) if depth[b, m] < max_depth
                     and children[m] < max_children and depth[b, m] < L]
            if not cand:
                raise ValueError("tree capacity exhausted")
            par = cand[rng.integers(len(cand))]
            children[par] += 1
            used = set()
            m = par
            while m != N:
                used.add(int(pos[b, m]))
                m = parent[b, m] if parent[b, m] >= 0 else N
            free = [s for s in range(L) if s not in used]
            pos[b, n] = free[rng.integers(len(free))]
            parent[b, n] = -1 if par == N else par
            depth[b, n] = 1 if par == N else depth[b, par] + 1
    return parent, pos, depth


def tree_inputs(B, N, V, dtype="bf16", seed=3, L=32, max_depth=8, max_children=4,
                p_match=0.8, device="cpu") -> TreeInputs:
    parent, pos, depth = random_trees(B, N, L, max_depth, max_children, seed)
    g = _gen(seed, device)
    logits = _normal((B, N, V), 2.0, g, device).to(_TORCH_DTYPE[dtype])
    tok = _pick_tokens(logits, p_match, g, device)
    t = lambda a: torch.as_tensor(a, dtype=torch.int32, device=device)
    return TreeInputs(logits, t(parent), t(pos), tok, depth)


@dataclasses.dataclass
class PackedInputs:
    logits: torch.Tensor             # [B, K+W, V]
    prev_draft: torch.Tensor         # [B, K-1] int32
    prev_len: torch.Tensor           # [B] int32
    prev_q_at_draft: torch.Tensor    # [B, K-1] fp32 (T > 0)
    prev_draft_logits: torch.Tensor  # [B, W, V] (T > 0)
    prev_q_offset: torch.Tensor      # [B] int32


def packed_inputs(B, K, W, V, dtype="bf16", seed=4, T=0.0, p_match=0.8, device="cpu",
                  sigma=0.5) -> PackedInputs:
    """A Packed-SS state after a previous call that advanced by a_prev ~ U{1..W}:
    the previous draft has W - a_prev tokens (capped at K - 1)."""
    g = _gen(seed, device)
    dt = _TORCH_DTYPE[dtype]
    lg32 = _normal((B, K + W, V), 2.0, g, device)
    a_prev = torch.randint(1, W + 1, (B,), generator=g, device=device)
    prev_len = torch.clamp(W - a_prev, max=K - 1).to(torch.int32)
    logits = lg32.to(dt)
    if T == 0.0:
        pd = _pick_tokens(logits[:, :K - 1], p_match, g, device) if K > 1 else \
            torch.zeros((B, 0), dtype=torch.int32, device=device)
        pq = torch.ones((B, K - 1), dtype=torch.float32, device=device)
        pdl = torch.empty((B, W, V), dtype=dt, device=device)[:0]
        del lg32
        return PackedInputs(logits, pd, prev_len, pq, pdl, a_prev.to(torch.int32))
    # previous drafter rows: row a_prev + i is the verify row i plus noise
    prev32 = _normal((B, W, V), 2.0, g, device)
    idx = torch.arange(W, device=device)[None, :] - a_prev[:, None]          # [B, W]
    src = idx.clamp(0, K - 1)
    use = (idx >= 0) & (idx < K)
    gathered = torch.gather(lg32[:, :K], 1, src[:, :, None].expand(B, W, V))
    prev32 = torch.where(use[:, :, None], gathered + _normal((B, W, V), sigma, g, device),
                         prev32)
    del gathered, lg32
    pdl = prev32.to(dt)
    del prev32
    # the retained draft d_i ~ Q_i = softmax(row a_prev + i / T), and Q_i(d_i)
    rows = torch.gather(pdl, 1, (a_prev[:, None] + torch.arange(K - 1, device=device)[None])
                        .clamp(max=W - 1)[:, :, None].expand(B, K - 1, V))
    pd = _draw_from_logits(rows, T, g, device) if K > 1 else \
        torch.zeros((B, 0), dtype=torch.int32, device=device)
    probs = torch.softmax(rows.float() / T, dim=-1)
    pq = torch.gather(probs, 2, pd.long()[:, :, None])[:, :, 0].contiguous()
    del rows, probs
    return PackedInputs(logits, pd, prev_len, pq, pdl, a_prev.to(torch.int32))


def to_numpy_logits(t: torch.Tensor) -> np.ndarray:
    """fp32 -> float32 array; bf16 -> uint16 array of the raw bit patterns."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)


@dataclasses.dataclass
class SpotInputs:
    state_logits: torch.Tensor  # [B, 1+N, L, V]
    parent: torch.Tensor        # [B, N] int32, -1 = child of the root
    node_pos: torch.Tensor      # [B, N] int32, a masked position of the parent's state
    node_tok: torch.Tensor      # [B, N] int32
    root_mask: torch.Tensor     # [B] int64, bit s = position s masked at the root
    masks: np.ndarray           # [B, 1+N] host-side masks of every state


def spot_trees(B, N, L, max_depth=8, max_children=4, seed=5, root_masked=None):
    """Random SPOT draft trees (host numpy): the root state has root_masked
    masked positions (all L by default, else a uniform subset); node n picks
    a uniform parent among the root and the earlier nodes that have a masked
    position left, depth below max_depth and fewer than max_children
    children, and commits at a uniform masked position of that parent's
    state."""
    rng = np.random.default_rng(seed)
    parent = np.full((B, N), -1, np.int32)
    pos = np.zeros((B, N), np.int32)
    masks = np.zeros((B, N + 1), np.uint64)
    k = L if root_masked is None else root_masked
    for b in range(B):
        m0 = 0
        for s in rng.choice(L, size=k, replace=False):
            m0 |= 1 << int(s)
        masks[b, 0] = m0
        depth = np.zeros(N + 1, np.int64)
        children = np.zeros(N + 1, np.int64)
        for n in range(N):
            cand = [a for a in range(n + 1) if int(masks[b, a]) != 0 and depth[a] < max_depth
                    and children[a] < max_children]
            a = cand[rng.integers(len(cand))]
            free = [s for s in range(L) if (int(masks[b, a]) >> s) & 1]
            s = free[rng.integers(len(free))]
            parent[b, n] = a - 1
            pos[b, n] = s
            masks[b, n + 1] = int(masks[b, a]) & ~(1 << s)
            depth[n + 1] = depth[a] + 1
            children[a] += 1
    return parent, pos, masks


def spot_inputs(B, N, L, V, dtype="bf16", seed=5, max_depth=8, max_children=4, p_match=0.8,
                root_masked=None, device="cpu") -> SpotInputs:
    """SPOT workload: rows N(0, 2^2) for every (state, position); node tokens
    = the largest entry of the parent state's row at the node's position with
    probability p_match, else a uniform other id."""
    parent, pos, masks = spot_trees(B, N, L, max_depth, max_children, seed, root_masked)
    g = _gen(seed, device)
    logits = _normal((B, N + 1, L, V), 2.0, g, device).to(_TORCH_DTYPE[dtype])
    t = lambda a: torch.as_tensor(a, dtype=torch.int32, device=device)
    par_state = torch.as_tensor(parent.astype(np.int64) + 1, device=device)
    rows = logits[torch.arange(B, device=device)[:, None], par_state,
                  torch.as_tensor(pos.astype(np.int64), device=device)] if N > 0 else None
    tok = _pick_tokens(rows, p_match, g, device) if N > 0 else \
        torch.zeros((B, 0), dtype=torch.int32, device=device)
    rm = torch.as_tensor(masks[:, 0].astype(np.int64), device=device)
    return SpotInputs(logits, t(parent), t(pos), tok, rm, masks)


@dataclasses.dataclass
class AnyOrderInputs:
    logits: torch.Tensor   # [B, Kv + W, V]
    u: torch.Tensor        # [B] int32
    win_pos: torch.Tensor  # [B, W] int32, ascending output positions
    order: torch.Tensor    # [B, W] int32, window index of each rank
    draft: torch.Tensor    # [B, W] int32, -1 = no draft
    end_pos: torch.Tensor  # [B] int32


def anyorder_inputs(B, Kv, W, V, dtype="bf16", seed=6, p_draft=0.9, p_match=0.8, ragged=False,
                    device="cpu") -> AnyOrderInputs:
    """Any-order Packed-SS state: u unresolved window positions (W, or uniform
    in 1..W when ragged) at ascending output positions with random gaps, a
    random rank order, a draft token at each position with probability
    p_draft -- at rank r the largest entry of verify row r with probability
    p_match, else a uniform other id -- and rows N(0, 2^2)."""
    rng = np.random.default_rng(seed)
    g = _gen(seed, device)
    logits = _normal((B, Kv + W, V), 2.0, g, device).to(_TORCH_DTYPE[dtype])
    best = logits[:, :Kv].float().argmax(-1).cpu().numpy()
    u = rng.integers(1, W + 1, B) if ragged else np.full(B, W)
    wp = np.full((B, W), -1, np.int32)
    od = np.full((B, W), -1, np.int32)
    dr = np.full((B, W), -1, np.int32)
    for b in range(B):
        n = int(u[b])
        wp[b, :n] = np.sort(rng.choice(np.arange(1, 4 * W + 1), n, replace=False))
        od[b, :n] = rng.permutation(n)
        for r in range(n):
            if rng.random() < p_draft:
                if r < Kv and rng.random() < p_match:
                    dr[b, od[b, r]] = best[b, r]
                else:
                    dr[b, od[b, r]] = int(rng.integers(V))
    t = lambda a: torch.as_tensor(a, dtype=torch.int32, device=device)
    return AnyOrderInputs(logits, t(u), t(wp), t(od), t(dr), t(np.full(B, 10 ** 6)))


@dataclasses.dataclass
class PackedTopkInputs:
    prev_logits: torch.Tensor   # [B, K+W, V] the previous call's rows
    logits: torch.Tensor        # [B, K+W, V] this call's rows
    a_prev: torch.Tensor        # [B] int32: the previous call's stopping index, 1..W


def packed_topk_inputs(B, K, W, V, dtype="bf16", seed=7, sigma=0.3, device="cpu"):
    """Two consecutive model calls of a Packed-SS run: rows N(0, 2^2); this
    call's verify row i repeats the previous call's proposal row a_prev + i
    plus N(0, sigma^2) noise (a drafter that saw the same context), with
    a_prev ~ U{1..W}.  The truncated lists and drafts of the previous call
    are the step's own outputs on prev_logits (see packed_state_from)."""
    g = _gen(seed, device)
    dt = _TORCH_DTYPE[dtype]
    prev = _normal((B, K + W, V), 2.0, g, device)
    cur = _normal((B, K + W, V), 2.0, g, device)
    a_prev = torch.randint(1, W + 1, (B,), generator=g, device=device)
    idx = torch.arange(K, device=device)[None, :] + a_prev[:, None]           # [B, K]
    use = idx < W
    src = torch.gather(prev[:, K:], 1, idx.clamp(max=W - 1)[:, :, None].expand(B, K, V))
    cur[:, :K] = torch.where(use[:, :, None], src + _normal((B, K, V), sigma, g, device),
                             cur[:, :K])
    del src
    return PackedTopkInputs(prev.to(dt), cur.to(dt), a_prev.to(torch.int32))


def packed_state_from(next_draft, commit_len, q_ids, q_probs, a_prev, K, W):
    """The inputs of the next truncated Packed-SS call when the previous call
    (outputs next_draft, commit_len, q_ids, q_probs; numpy or torch) is taken
    to have stopped at a_prev instead of its own commit_len: the draft is
    z_{a_prev + i}, i < min(W - a_prev, K - 1), and Q_{t-1}^(i) is list
    a_prev + i (offset a_prev).  Pure indexing; a_prev >= commit_len."""
    lib = torch if isinstance(next_draft, torch.Tensor) else np
    B = next_draft.shape[0]
    n = lib.clip(W - a_prev, 0, K - 1) if lib is np else torch.clamp(W - a_prev, 0, K - 1)
    i = lib.arange(K - 1)[None, :] if lib is np else torch.arange(K - 1,
                                                                  device=next_draft.device)[None]
    src = (a_prev - commit_len)[:, None] + i
    valid = i < n[:, None]
    if lib is np:
        d = np.take_along_axis(next_draft, np.clip(src, 0, W - 1), 1)
        prev_draft = np.where(valid, d, 0).astype(np.int32)
        return dict(prev_draft=prev_draft, prev_len=n.astype(np.int32),
                    prev_q_offset=a_prev.astype(np.int32), prev_q_ids=q_ids.astype(np.int32),
                    prev_q_probs=q_probs.astype(np.float32))
    d = torch.gather(next_draft, 1, src.clamp(0, W - 1).long())
    prev_draft = torch.where(valid, d, torch.zeros_like(d)).to(torch.int32).contiguous()
    return dict(prev_draft=prev_draft, prev_len=n.to(torch.int32).contiguous(),
                prev_q_offset=a_prev.to(torch.int32).contiguous(),
                prev_q_ids=q_ids.to(torch.int32).contiguous(),
                prev_q_probs=q_probs.to(torch.float32).contiguous())

