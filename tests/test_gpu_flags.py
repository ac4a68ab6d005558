"""GPU parity on decisions that fall within 1e-9 of their thresholds.

The inputs are built on the host with the oracle (flag_cases.py) so that some
acceptance tests and Gumbel-max draws are near ties; both sides must count
each one in `flags` (the counts are compared exactly and must be non-zero),
and every sequence that neither side flags must still match bit for bit.
The library reaches these decisions on its fast fp32 path, finds them inside
their error bound and settles them on the fp64 path."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from flag_cases import near_threshold_acceptance, near_tie_key, near_tie_row
from gpu_util import DEV, RTOL, assert_float_close, compare_sample, cpu

pytestmark = pytest.mark.gpu

V = 4096


@pytest.fixture(scope="module")
def dbv():
    import draft_block_verification_gb300 as m
    m.build()
    m.lib()
    oracle.build()
    return m


def _t(a, dtype=None):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def test_flagged_sample_decisions(dbv):
    """Six sequences, K = 2: near-threshold acceptance at position 0 (above and
    below u), at position 1 after a certain accept, a near-tie bonus draw after
    two certain accepts, and two ordinary sequences."""
    rng = np.random.default_rng(17)
    B, K, seed = 6, 2, 23
    pos = np.array([10, 20, 30, 0, 50, 60], np.int64)
    tg = rng.standard_normal((B, K + 1, V)).astype(np.float32) * 2
    dr = (tg[:, :K] + 0.5 * rng.standard_normal((B, K, V))).astype(np.float32)
    ids = rng.integers(0, V, (B, K)).astype(np.int32)
    u = lambda b, i: oracle.uniform(oracle.key(seed, oracle.ST_ACCEPT, b, int(pos[b]) + i, 0), 0)
    # sequences 0, 1: position 0 within 4e-10 of u (accepted / rejected)
    for b, sign in ((0, 1), (1, -1)):
        tg[b, 0], dr[b, 0], _ = near_threshold_acceptance(V, u(b, 0), sign, rng)
        ids[b, 0] = 7
    # sequence 2: position 0 certain (p = q, alpha = 1), position 1 near u
    dr[2, 0] = tg[2, 0]
    tg[2, 1], dr[2, 1], _ = near_threshold_acceptance(V, u(2, 1), 1, rng)
    ids[2, 1] = 7
    # sequence 3: both tests certain, the bonus draw (row 2) a near tie
    dr[3] = tg[3, :K]
    p3, a, b = near_tie_key(lambda q: oracle.key(seed, oracle.ST_SAMPLE, 3, q + K, 0), V)
    pos[3] = p3
    tg[3, K], _ = near_tie_row(oracle.key(seed, oracle.ST_SAMPLE, 3, p3 + K, 0), V, a, b, 1.0, 1)
    out = dbv.sv_verify_sample(_t(tg), _t(dr), _t(ids), T_p=1.0, T_q=1.0, seed=seed,
                               pos_base=_t(pos), want_tv=True)
    dbv.default_handle().sync_status()
    ref = oracle.verify_sample(tg, dr, ids, T_p=1.0, T_q=1.0, seed=seed, pos_base=pos)
    assert ref["flags"][:4].tolist() == [1, 1, 1, 1], ref["flags"]
    assert ref["flags"][4:].tolist() == [0, 0]
    n = compare_sample(out, ref, "f32")
    assert n == 2
    # the flagged decisions still come out as they were aimed, on both sides
    for acc in (cpu(out["accept_len"]), ref["accept_len"]):
        assert acc[0] >= 1 and acc[1] == 0 and acc[2] == 2 and acc[3] == 2, acc


def test_flagged_tree_nodes(dbv):
    """Three trees of 8 nodes at T = 1: a near-tie coupled-noise draw at one node
    of trees 0 and 1 (the runner-up ahead / behind), tree 2 ordinary."""
    B, N, seed = 3, 8, 29
    parent, npos, _ = datagen.random_trees(B, N, L=8, max_depth=4, max_children=3, seed=4)
    rng = np.random.default_rng(5)
    rows = (rng.standard_normal((B, N, V)) * 2).astype(np.float32)
    pos_base = np.array([0, 0, 7], np.int64)
    for b, node, sign, start in ((0, 0, 1, 0), (1, 3, -1, 3000)):
        p, a, c = near_tie_key(
            lambda q: oracle.key(seed, oracle.ST_TREE, b, q + int(npos[b, node]), 0), V,
            start=start)
        pos_base[b] = p
        k = oracle.key(seed, oracle.ST_TREE, b, p + int(npos[b, node]), 0)
        rows[b, node], _ = near_tie_row(k, V, a, c, 1.0, sign)
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    for b in range(B):  # each node's own winner, so that paths are deep
        for n in range(N):
            k = oracle.key(seed, oracle.ST_TREE, b, int(pos_base[b] + npos[b, n]), 0)
            tok[b, n] = oracle.gumbel_argmax(rows[b, n].astype(np.float64), k)[0]
    out = dbv.sv_verify_tree(_t(rows), _t(parent), _t(npos), _t(tok), T=1.0, seed=seed,
                             pos_base=_t(pos_base), max_depth=4)
    dbv.default_handle().sync_status()
    ref = oracle.verify_tree(rows, parent, npos, tok, T=1.0, seed=seed, pos_base=pos_base,
                             max_depth=4)
    assert (ref["flags"][:2] >= 1).all() and ref["flags"][2] == 0, ref["flags"]
    assert np.array_equal(cpu(out["flags"]), ref["flags"])
    for k in ("path_len", "path_nodes", "commit_count", "match"):
        assert np.array_equal(cpu(out[k])[2], ref[k][2]), k
    assert ref["path_len"][2] >= 1


def test_flagged_packed_proposal(dbv):
    """Packed-SS at T = 1 with an empty previous draft: a near-tie proposal draw
    at draft row 1 of sequence 0; sequence 1 ordinary."""
    B, K, W, seed, it = 2, 2, 3, 31, 5
    rng = np.random.default_rng(8)
    lg = (rng.standard_normal((B, K + W, V)) * 2).astype(np.float32)
    p0, a, c = near_tie_key(lambda q: oracle.key(seed, oracle.ST_DRAFT, 0, q + 1, it), V)
    pos = np.array([p0, 100], np.int64)
    lg[0, K + 1], _ = near_tie_row(oracle.key(seed, oracle.ST_DRAFT, 0, p0 + 1, it), V, a, c,
                                   1.0, 1)
    prev_len = np.zeros(B, np.int32)
    prev_draft = np.zeros((B, K - 1), np.int32)
    prev_q = np.ones((B, K - 1), np.float32)
    prev_rows = (rng.standard_normal((B, W, V)) * 2).astype(np.float32)
    off = np.ones(B, np.int32)
    out = dbv.sv_packed_step(_t(lg), K, W, _t(prev_draft), _t(prev_len),
                             prev_q_at_draft=_t(prev_q), prev_draft_logits=_t(prev_rows),
                             prev_q_offset=_t(off), T=1.0, seed=seed, it=it, pos_base=_t(pos))
    dbv.default_handle().sync_status()
    ref = oracle.packed_step(lg, K, W, prev_draft, prev_len, prev_q, prev_rows, off, T=1.0,
                             seed=seed, it=it, pos_base=pos)
    assert ref["flags"].tolist()[0] >= 1 and ref["flags"][1] == 0, ref["flags"]
    assert np.array_equal(cpu(out["flags"]), ref["flags"])
    for k in ("accept_len", "commit_len", "committed", "next_draft", "next_len"):
        assert np.array_equal(cpu(out[k])[1], ref[k][1]), k
    assert_float_close(cpu(out["confidence"]), ref["confidence"], RTOL["f32"], 0.0, "confidence")
