"""Helpers shared by the GPU parity tests (not collected as tests)."""
import numpy as np
import torch

import datagen
import oracle

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None
np_logits = datagen.to_numpy_logits

# Float tolerances of returned probabilities / log-sum-exps / TV, relative,
# by input dtype; TV also gets an absolute floor of 4e-6 (fp32 summation of up
# to 2^18 terms in a quantity near 1).
RTOL = {"f32": 1e-5, "bf16": 2e-3}
TV_ATOL = 4e-6


def bits_to_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def cpu(x):
    return x.detach().cpu().numpy()


def assert_float_close(got, ref, rtol, atol=0.0, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, what
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), "%s: NaN pattern differs" % what
    ok = ~nan_r
    err = np.abs(got[ok] - ref[ok])
    lim = rtol * np.abs(ref[ok]) + atol
    bad = err > lim
    assert not bad.any(), "%s: %d/%d outside tolerance, worst %.3g (ref %.6g got %.6g)" % (
        what, int(bad.sum()), bad.size, float(err.max()),
        float(ref[ok][np.argmax(err - lim)]), float(got[ok][np.argmax(err - lim)]))


def compare_sample(out, ref, dtype, want_tv=True):
    """Bit-exact decisions on every sequence neither side flagged; fp outputs
    within the dtype's tolerance everywhere."""
    fg, fr = cpu(out["flags"]), ref["flags"]
    assert np.array_equal(fg, fr), "flag counts differ"
    keep = fr == 0
    assert np.array_equal(cpu(out["accept_len"])[keep], ref["accept_len"][keep])
    assert np.array_equal(cpu(out["next_token"])[keep], ref["next_token"][keep])
    rt = RTOL[dtype]
    for k in ("p_at_draft", "q_at_draft", "lse_p", "lse_q"):
        if k in out:
            assert_float_close(cpu(out[k]), ref[k], rt, 0.0, k)
    if want_tv and "tv" in out:
        assert_float_close(cpu(out["tv"]), ref["tv"], rt, TV_ATOL, "tv")
    return int(keep.sum())


def craft_tree_tokens(node_logits_np, pos, T, seed, rng, p=0.8, pos_base=None):
    """node_tok: the oracle's own commitment at each node with probability p,
    else a uniform id (so that draft trees have deep accepted paths)."""
    B, N, V = node_logits_np.shape
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    Tf = oracle.f32(T)
    for b in range(B):
        pb = 0 if pos_base is None else int(pos_base[b])
        for n in range(N):
            if rng.random() >= p:
                continue
            x = bits_to_f64(node_logits_np[b, n])
            if T == 0.0:
                tok[b, n] = oracle.argmax(x)
            else:
                k = oracle.key(seed, oracle.ST_TREE, b, pb + int(pos[b, n]), 0)
                tok[b, n] = oracle.gumbel_argmax(x / Tf, k)[0]
    return tok


def craft_spot_tree(rows_np, root_mask, N, T, seed, rng, p=0.7, pos_base=None,
                    max_children=4):
    """A SPOT tree for given state rows [B, 1+N, L, V]: node n takes a uniform
    parent among the states with a masked position left and fewer than
    max_children children; with probability p it commits the oracle's own
    transition Phi of that parent state (so that paths are deep), else a
    uniform masked position and a uniform token.  Returns (parent, node_pos,
    node_tok) as int32 arrays [B, N]."""
    B, S, L, V = rows_np.shape
    parent = np.full((B, N), -1, np.int32)
    pos = np.zeros((B, N), np.int32)
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        masks = [int(root_mask[b])]
        kids = [0] * (N + 1)
        pb = 0 if pos_base is None else int(pos_base[b])
        for n in range(N):
            cand = [a for a in range(n + 1) if masks[a] and kids[a] < max_children]
            a = cand[rng.integers(len(cand))]
            if rng.random() < p:
                r = oracle.verify_spot(rows_np[b:b + 1, a:a + 1], np.zeros((1, 0)),
                                       np.zeros((1, 0)), np.zeros((1, 0)),
                                       np.array([masks[a]], np.uint64), T=T, seed=seed,
                                       pos_base=np.array([pb]))
                s, v = int(r["commit_pos"][0]), int(r["commit_tok"][0])
                # the row of state a at position s is row (b, a, s): the call above
                # saw it as sequence 0, so its noise key used sequence 0, not b
                if T > 0:
                    k = oracle.key(seed, oracle.ST_TREE, b, pb + s, 0)
                    v = oracle.gumbel_argmax(bits_to_f64(rows_np[b, a, s]) / oracle.f32(T), k)[0]
            else:
                free = [x for x in range(L) if (masks[a] >> x) & 1]
                s, v = free[rng.integers(len(free))], int(rng.integers(V))
            parent[b, n], pos[b, n], tok[b, n] = a - 1, s, v
            masks.append(masks[a] & ~(1 << s))
            kids[a] += 1
    return parent, pos, tok
