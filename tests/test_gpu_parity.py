"""GPU parity: every entry point, called through the C ABI, against the fp64
oracle on the same seeded inputs.  Integer results (accept lengths, tokens,
tree paths, next drafts) must be bit-exact on every sequence that neither
side flags as near-threshold; floats within the dtype's tolerance."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from gpu_util import (DEV, RTOL, assert_float_close, compare_sample, cpu, craft_spot_tree,
                      craft_tree_tokens, np_logits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbv():
    import draft_block_verification_gb300 as m
    m.build()
    m.lib()
    oracle.build()
    return m


def _g(t):
    return None if t is None else t.to(DEV)


# ------------------------------------------------------------------ greedy

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,K,V,ragged", [(3, 5, 4104, False), (2, 0, 64, False),
                                          (5, 8, 32000, True), (2, 32, 2056, True),
                                          (1, 3, 151936, False)])
def test_greedy_parity(dbv, dtype, B, K, V, ragged):
    gi = datagen.greedy_inputs(B, K, V, dtype=dtype, seed=B * 100 + K, ragged=ragged)
    acc, nxt = dbv.sv_verify_greedy(_g(gi.target), _g(gi.draft_ids), _g(gi.draft_len))
    r = oracle.verify_greedy(np_logits(gi.target), gi.draft_ids.numpy(), gi.draft_len.numpy())
    assert np.array_equal(cpu(acc), r["accept_len"])
    assert np.array_equal(cpu(nxt), r["next_token"])


def test_greedy_edges(dbv):
    V, K = 1024, 4
    # exact ties everywhere: the argmax is id 0
    t = torch.zeros((3, K + 1, V), dtype=torch.bfloat16)
    ids = torch.tensor([[0, 0, 0, 0], [0, 0, 5, 0], [7, 0, 0, 0]], dtype=torch.int32)
    acc, nxt = dbv.sv_verify_greedy(_g(t), _g(ids))
    assert cpu(acc).tolist() == [4, 2, 0] and cpu(nxt).tolist() == [0, 0, 0]
    # all accepted / all rejected with a bonus at the last id
    gi = datagen.greedy_inputs(4, K, V, dtype="bf16", seed=1, p_match=1.0)
    acc, nxt = dbv.sv_verify_greedy(_g(gi.target), _g(gi.draft_ids))
    assert cpu(acc).tolist() == [K] * 4
    gi = datagen.greedy_inputs(4, K, V, dtype="bf16", seed=2, p_match=0.0)
    acc, _ = dbv.sv_verify_greedy(_g(gi.target), _g(gi.draft_ids))
    assert cpu(acc).tolist() == [0] * 4
    t = torch.full((1, 2, V), -3.0)
    t[0, 1, V - 1] = 9.0
    acc, nxt = dbv.sv_verify_greedy(_g(t), _g(torch.zeros((1, 1), dtype=torch.int32)))
    assert (cpu(acc)[0], cpu(nxt)[0]) == (1, V - 1)


# ------------------------------------------------------------------ sampling

SAMPLE_CASES = [
    # dtype, B, K, V, mode, lam, Tp, Tq, sigma, ragged
    ("bf16", 8, 6, 8200, 0, 1.0, 1.0, 1.0, 0.5, False),
    ("f32", 6, 5, 4100, 0, 1.0, 0.7, 0.7, 0.5, True),
    ("bf16", 6, 7, 12288, 1, 2.0, 1.0, 1.0, 1.0, False),
    ("bf16", 6, 7, 12288, 1, 8.0, 0.7, 0.7, 0.25, False),
    ("bf16", 5, 4, 6152, 2, 0.5, 1.0, 1.0, 1.0, True),
    ("f32", 4, 3, 2048, 2, 0.875, 1.3, 0.9, 1.0, False),
    ("bf16", 3, 32, 2056, 0, 1.0, 1.0, 1.0, 0.5, True),
    ("bf16", 4, 0, 1024, 0, 1.0, 1.0, 1.0, 0.5, False),
    # modified Cactus: KL budget delta = lam
    ("bf16", 6, 7, 12288, 3, 0.05, 1.0, 1.0, 1.0, False),
    ("f32", 5, 4, 4100, 3, 0.5, 0.7, 0.7, 1.0, True),
    ("bf16", 4, 5, 8200, 3, 3.0, 1.0, 1.0, 0.5, False),
    ("bf16", 4, 5, 8200, 3, 0.0, 1.0, 1.0, 0.5, True),
    # enough rows for whole-row units (64 x 13 >= 4 x 152): rows of several
    # stages with a ragged tail, the TV kernel over whole rows
    ("bf16", 64, 6, 12296, 1, 2.0, 1.0, 1.0, 1.0, True),
    ("f32", 64, 6, 6148, 0, 1.0, 0.7, 0.7, 0.5, True),
    ("bf16", 64, 6, 12296, 3, 0.2, 1.0, 1.0, 0.5, False),
]


@pytest.mark.parametrize("dtype,B,K,V,mode,lam,Tp,Tq,sigma,ragged", SAMPLE_CASES)
def test_sample_parity(dbv, dtype, B, K, V, mode, lam, Tp, Tq, sigma, ragged):
    si = datagen.sample_inputs(B, K, V, dtype=dtype, seed=K * 7 + B, sigma=sigma, T=Tq,
                               ragged=ragged)
    pos = torch.arange(B, dtype=torch.int64) * 37 + 5
    out = dbv.sv_verify_sample(_g(si.target), _g(si.draft), _g(si.draft_ids),
                               _g(si.draft_len), T_p=Tp, T_q=Tq, mode=mode, lam=lam, seed=99,
                               pos_base=_g(pos), want_tv=True)
    ref = oracle.verify_sample(np_logits(si.target), np_logits(si.draft), si.draft_ids.numpy(),
                               si.draft_len.numpy(), T_p=Tp, T_q=Tq, mode=mode, lam=lam, seed=99,
                               pos_base=pos.numpy())
    compare_sample(out, ref, dtype)
    dbv.default_handle().sync_status()


@pytest.mark.parametrize("dtype,mode,lam", [("bf16", 0, 1.0), ("f32", 0, 1.0), ("bf16", 3, 0.2),
                                            ("f32", 3, 1.5)])
def test_sample_fp64_path(dbv, dtype, mode, lam):
    """Force every sequence through the fp64 path; it must agree too."""
    si = datagen.sample_inputs(10, 6, 4104, dtype=dtype, seed=5, sigma=1.0, ragged=True)
    h = dbv.Handle()
    try:
        h.set_option(dbv.SV_OPT_FORCE_RESCUE, 1)
        before = h.rescue_count()
        out = dbv.sv_verify_sample(_g(si.target), _g(si.draft), _g(si.draft_ids),
                                   _g(si.draft_len), mode=mode, lam=lam, seed=3, want_tv=True,
                                   handle=h)
        h.sync_status()
        assert h.rescue_count() - before == 10
    finally:
        h.close()
    ref = oracle.verify_sample(np_logits(si.target), np_logits(si.draft), si.draft_ids.numpy(),
                               si.draft_len.numpy(), mode=mode, lam=lam, seed=3)
    compare_sample(out, ref, dtype)


def test_sample_cactus_zero_budget_is_lossless(dbv):
    """The modified Cactus rule with delta = 0 gives the lossless results."""
    si = datagen.sample_inputs(12, 8, 8200, dtype="bf16", seed=44, sigma=1.0, ragged=True)
    args = (_g(si.target), _g(si.draft), _g(si.draft_ids), _g(si.draft_len))
    a = dbv.sv_verify_sample(*args, mode=3, lam=0.0, seed=6, want_tv=True)
    b = dbv.sv_verify_sample(*args, mode=0, seed=6, want_tv=True)
    for k in a:
        assert torch.equal(a[k].nan_to_num(), b[k].nan_to_num()), k


def test_sample_error_model(dbv):
    """The fp32 log-sum-exp error bound used to certify decisions holds: every
    returned p(d) is within the bound of the fp64 value."""
    si = datagen.sample_inputs(16, 8, 32768, dtype="bf16", seed=8, sigma=0.5)
    out = dbv.sv_verify_sample(_g(si.target), _g(si.draft), _g(si.draft_ids), seed=1)
    ref = oracle.verify_sample(np_logits(si.target), np_logits(si.draft), si.draft_ids.numpy(),
                               seed=1, want_tv=False)
    # the streamed log-sum-exp bound: ex2 error, exponent rounding of terms
    # within 2^-24 of the max, the weight of smaller terms, and 2^-24 per fp32
    # addition (a summation depth of 64 covers this launch)
    n, u, ln2 = 32768, 2.0**-24, 0.6931471805599453
    near = 2.0**-21 + 2 * ln2 * u * 24
    mid = 2.0**-21 + 2 * ln2 * u * 48
    eps = 2 * 2.0**-21 + near + 2 * n * u * mid + 2 * n * 2.0**-48 + 1.01 * 64 * u
    # p(d) = exp(x_d - L_p): its relative error is that of exp(L_p), plus the
    # fp32 rounding of the returned value
    bound = eps + 2.0**-23
    rel = np.abs(cpu(out["p_at_draft"]).astype(np.float64) / ref["p_at_draft"] - 1.0)
    assert np.all(rel <= bound), float((rel - bound).max())


def test_sample_deterministic_and_streams(dbv):
    si = datagen.sample_inputs(8, 5, 4104, dtype="bf16", seed=12)
    args = (_g(si.target), _g(si.draft), _g(si.draft_ids))
    a = dbv.sv_verify_sample(*args, seed=4, want_tv=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = dbv.sv_verify_sample(*args, seed=4, want_tv=True, stream=s)
    s.synchronize()
    for k in a:
        assert torch.equal(a[k].nan_to_num(), b[k].nan_to_num()), k


def test_sample_full_size_lossless(dbv):
    """The lossless T = 1 workload at full size: B = 64, K = 16, V = 128256 bf16."""
    c = datagen.CONFIGS["lossless_t1"]
    si = datagen.sample_inputs(c["B"], c["K"], c["V"], dtype="bf16", seed=c["seed"],
                               sigma=c["sigma"], T=c["T"], device=DEV)
    out = dbv.sv_verify_sample(si.target, si.draft, si.draft_ids, seed=c["seed"])
    ref = oracle.verify_sample(np_logits(si.target), np_logits(si.draft), cpu(si.draft_ids),
                               seed=c["seed"], want_tv=False)
    n = compare_sample(out, ref, "bf16", want_tv=False)
    assert n >= c["B"] - 1


@pytest.mark.parametrize("sigma,T,mode,lam", [(1.0, 0.7, 1, 4.0), (0.25, 1.0, 2, 0.75),
                                            (1.0, 1.0, 3, 0.1)])
def test_sample_full_size_lenient(dbv, sigma, T, mode, lam):
    """Two points of the lenient sweep at full size (B = 128, K = 16, V = 151936)."""
    c = datagen.CONFIGS["lenient_sweep"]
    si = datagen.sample_inputs(c["B"], c["K"], c["V"], dtype="bf16", seed=c["seed"],
                               sigma=sigma, T=T, device=DEV)
    out = dbv.sv_verify_sample(si.target, si.draft, si.draft_ids, T_p=T, T_q=T, mode=mode,
                               lam=lam, seed=c["seed"], want_tv=True)
    ref = oracle.verify_sample(np_logits(si.target), np_logits(si.draft), cpu(si.draft_ids),
                               T_p=T, T_q=T, mode=mode, lam=lam, seed=c["seed"])
    compare_sample(out, ref, "bf16")


# ------------------------------------------------------------------ tree

@pytest.mark.parametrize("T", [0.0, 1.0, 0.7])
@pytest.mark.parametrize("B,N,V,md", [(4, 20, 5000, 8), (2, 64, 2048, 8), (3, 1, 1024, 1),
                                      (2, 30, 4096, 2)])
def test_tree_parity(dbv, T, B, N, V, md):
    ti = datagen.tree_inputs(B, N, V, dtype="bf16", seed=N + B, L=16, max_depth=8)
    pos_base = np.arange(B, dtype=np.int64) * 100
    tok = craft_tree_tokens(np_logits(ti.node_logits), ti.node_pos.numpy(), T, 21,
                            np.random.default_rng(N), pos_base=pos_base)
    out = dbv.sv_verify_tree(_g(ti.node_logits), _g(ti.parent), _g(ti.node_pos),
                             _g(torch.from_numpy(tok)), T=T, seed=21,
                             pos_base=_g(torch.from_numpy(pos_base)), max_depth=md)
    ref = oracle.verify_tree(np_logits(ti.node_logits), ti.parent.numpy(), ti.node_pos.numpy(),
                             tok, T=T, seed=21, pos_base=pos_base, max_depth=md)
    assert np.array_equal(cpu(out["flags"]), ref["flags"])
    keep = ref["flags"] == 0
    for k in ("path_len", "commit_count", "path_nodes", "match"):
        assert np.array_equal(cpu(out[k])[keep], ref[k][keep]), k
    assert ref["path_len"].max() >= 1


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tree_full_size(dbv, T):
    """The tree workload at full size: 32 trees x 64 nodes, V = 151936 bf16."""
    c = datagen.CONFIGS["tree"]
    ti = datagen.tree_inputs(c["B"], c["N"], c["V"], dtype="bf16", seed=c["seed"], L=c["L"],
                             max_depth=c["max_depth"], max_children=c["max_children"],
                             device=DEV)
    # the drafter's tokens: at T = 0 the workload's own (argmax w.p. 0.8); at
    # T > 0 the oracle's coupled-noise winner of each node w.p. 0.8, so that the
    # trees hold deep accepted paths at full vocabulary size too
    # (the first 8 trees; crafting costs the oracle a full row per node)
    tok = ti.node_tok
    if T > 0:
        S = 8
        crafted = craft_tree_tokens(np_logits(ti.node_logits[:S]), cpu(ti.node_pos[:S]), T,
                                    c["seed"], np.random.default_rng(5))
        tok = tok.clone()
        tok[:S] = torch.from_numpy(crafted).to(DEV)
    out = dbv.sv_verify_tree(ti.node_logits, ti.parent, ti.node_pos, tok, T=T,
                             seed=c["seed"], max_depth=8)
    ref = oracle.verify_tree(np_logits(ti.node_logits), cpu(ti.parent), cpu(ti.node_pos),
                             cpu(tok), T=T, seed=c["seed"], max_depth=8)
    keep = ref["flags"] == 0
    assert np.array_equal(cpu(out["flags"]), ref["flags"])
    for k in ("path_len", "path_nodes", "match", "commit_count"):
        assert np.array_equal(cpu(out[k])[keep], ref[k][keep]), k
    assert ref["path_len"][:8].max() >= 2 and ref["match"][:8].mean() > 0.5


# ------------------------------------------------------------------ SPOT

SPOT_KEYS = ("path_len", "path_nodes", "commit_count", "commit_pos", "commit_tok", "match",
             "state_pos", "state_tok")


def _spot_both(dbv, rows, parent, pos, tok, root_mask, T, seed, pos_base, md):
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    out = dbv.sv_verify_spot(rows.to(DEV), g(parent), g(pos), g(tok),
                             g(root_mask.astype(np.int64)), T=T, seed=seed, pos_base=g(pos_base),
                             max_depth=md)
    ref = oracle.verify_spot(np_logits(rows), parent, pos, tok, root_mask.astype(np.uint64),
                             T=T, seed=seed, pos_base=pos_base, max_depth=md)
    return out, ref


def _compare_spot(out, ref):
    assert np.array_equal(cpu(out["flags"]), ref["flags"])
    keep = ref["flags"] == 0
    for k in SPOT_KEYS:
        assert np.array_equal(cpu(out[k])[keep], ref[k][keep]), k


@pytest.mark.parametrize("T", [0.0, 1.0, 0.7])
@pytest.mark.parametrize("dtype,B,N,L,V,masked", [("bf16", 4, 10, 8, 2056, None),
                                                  ("f32", 3, 20, 16, 4100, 11),
                                                  ("bf16", 2, 0, 5, 1024, None),
                                                  ("bf16", 2, 64, 32, 1032, None)])
def test_spot_parity(dbv, T, dtype, B, N, L, V, masked):
    g = torch.Generator().manual_seed(N * 7 + L)
    rows = (torch.randn((B, N + 1, L, V), generator=g) * 2).to(
        torch.bfloat16 if dtype == "bf16" else torch.float32)
    rng = np.random.default_rng(N + L)
    root = np.zeros(B, np.uint64)
    for b in range(B):
        for x in rng.choice(L, size=L if masked is None else masked, replace=False):
            root[b] |= np.uint64(1 << int(x))
    pos_base = np.arange(B, dtype=np.int64) * 64 + 9
    parent, pos, tok = craft_spot_tree(np_logits(rows), root, N, T, 17, rng, pos_base=pos_base)
    md = max(N, 1)
    out, ref = _spot_both(dbv, rows, parent, pos, tok, root, T, 17, pos_base, md)
    _compare_spot(out, ref)
    if N >= 10:
        assert ref["path_len"].max() >= 2


def test_spot_confidence_ties_and_unmasked_rows(dbv):
    """Equal rows at two masked positions: the lower position wins, unflagged;
    a huge peak at an unmasked position is never read."""
    L, V = 6, 1024
    rows = torch.randn((1, 1, L, V)) * 2
    rows[0, 0, 4] = rows[0, 0, 1]
    rows[0, 0, 1, 3] = 12.0
    rows[0, 0, 4, 3] = 12.0
    rows[0, 0, 2, 5] = 1000.0  # unmasked below
    root = np.array([0b110011], np.uint64)
    e = np.zeros((1, 0), np.int32)
    out, ref = _spot_both(dbv, rows, e, e, e, root, 0.0, 1, np.zeros(1, np.int64), 1)
    _compare_spot(out, ref)
    assert int(cpu(out["commit_pos"])[0]) == 1 and int(cpu(out["flags"])[0]) == 0


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_spot_full_size(dbv, T):
    """The SPOT workload at full size: 32 trees of 8 drafted states over a
    32-position block, V = 151936 bf16 (the first 8 trees follow the target's
    own transitions with probability 0.7, so that paths are deep)."""
    c = datagen.CONFIGS["spot"]
    si = datagen.spot_inputs(c["B"], c["N"], c["L"], c["V"], dtype="bf16", seed=c["seed"],
                             device=DEV)
    rows_np = np_logits(si.state_logits)
    root = cpu(si.root_mask).astype(np.uint64)
    parent, pos, tok = cpu(si.parent), cpu(si.node_pos), cpu(si.node_tok)
    S = 8
    p8, q8, t8 = craft_spot_tree(rows_np[:S], root[:S], c["N"], T, c["seed"],
                                 np.random.default_rng(3))
    parent, pos, tok = parent.copy(), pos.copy(), tok.copy()
    parent[:S], pos[:S], tok[:S] = p8, q8, t8
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    out = dbv.sv_verify_spot(si.state_logits, g(parent), g(pos), g(tok), si.root_mask, T=T,
                             seed=c["seed"], max_depth=c["N"])
    ref = oracle.verify_spot(rows_np, parent, pos, tok, root, T=T, seed=c["seed"],
                             max_depth=c["N"])
    _compare_spot(out, ref)
    assert ref["path_len"][:S].max() >= 2


def test_spot_position_not_masked_is_latched(dbv):
    rows = torch.randn((2, 3, 4, 1024), device=DEV)
    par = torch.tensor([[-1, 0], [-1, 0]], dtype=torch.int32, device=DEV)
    pos = torch.tensor([[1, 1], [1, 2]], dtype=torch.int32, device=DEV)  # tree 0: 1 twice
    tok = torch.zeros((2, 2), dtype=torch.int32, device=DEV)
    root = torch.full((2,), 0b1111, dtype=torch.int64, device=DEV)
    h = dbv.Handle()
    try:
        dbv.sv_verify_spot(rows, par, pos, tok, root, handle=h)
        with pytest.raises(dbv.SVError) as e:
            h.sync_status()
        assert e.value.status == dbv.SV_ERR_DEVICE_BOUNDS
        pos[0, 1] = 3
        out = dbv.sv_verify_spot(rows, par, pos, tok, root, handle=h)
        h.sync_status()
        ref = oracle.verify_spot(np_logits(rows), cpu(par), cpu(pos), cpu(tok),
                                 cpu(root).astype(np.uint64))
        _compare_spot(out, ref)
    finally:
        h.close()


# ------------------------------------------------------------------ any-order Packed-SS

AO_KEYS = ("accept_len", "commit_len", "commit_pos", "commit_tok", "end_pos", "next_draft")


def _anyorder_both(dbv, ai, Kv, W, eos=-1, end=None):
    end = ai.end_pos if end is None else end
    out = dbv.sv_packed_anyorder_step(ai.logits.to(DEV), Kv, W, ai.u.to(DEV), ai.win_pos.to(DEV),
                                      ai.order.to(DEV), ai.draft.to(DEV), end.to(DEV), eos_id=eos)
    ref = oracle.packed_anyorder_step(np_logits(ai.logits), Kv, W, cpu(ai.u), cpu(ai.win_pos),
                                      cpu(ai.order), cpu(ai.draft), cpu(end), eos_id=eos)
    return out, ref


def _compare_anyorder(out, ref, dtype):
    for k in AO_KEYS:
        assert np.array_equal(cpu(out[k]), ref[k]), k
    assert_float_close(cpu(out["score"]), ref["score"], RTOL[dtype], 0.0, "score")


@pytest.mark.parametrize("dtype,B,Kv,W,V,ragged,p_draft", [
    ("bf16", 6, 8, 8, 4104, True, 0.9), ("f32", 4, 5, 5, 2048, False, 1.0),
    ("bf16", 3, 32, 32, 1032, True, 0.95), ("bf16", 5, 1, 1, 1024, False, 0.5),
    ("bf16", 4, 6, 6, 2056, True, 0.0)])
def test_anyorder_parity(dbv, dtype, B, Kv, W, V, ragged, p_draft):
    ai = datagen.anyorder_inputs(B, Kv, W, V, dtype=dtype, seed=B * 10 + W, p_draft=p_draft,
                                 ragged=ragged)
    out, ref = _anyorder_both(dbv, ai, Kv, W)
    _compare_anyorder(out, ref, dtype)
    # an accepted EOS lowers the end: the first accepted token of sequence 0
    # becomes EOS (window positions lie in 1..4W, so every pair was within
    # the end before)
    eos = int(ref["commit_tok"][0, 0])
    first = int(ref["commit_pos"][0, 0])
    out, ref = _anyorder_both(dbv, ai, Kv, W, eos=eos)
    _compare_anyorder(out, ref, dtype)
    assert ref["end_pos"][0] <= first


@pytest.mark.parametrize("which", ["not_a_permutation", "too_few_rows"])
def test_anyorder_bad_inputs_are_latched(dbv, which):
    ai = datagen.anyorder_inputs(2, 4, 4, 1024, dtype="bf16", seed=3, p_draft=1.0)
    Kv = 4
    if which == "not_a_permutation":
        ai.order[1, 1] = ai.order[1, 0]
    else:
        Kv = 2  # all four positions have drafts: min(kappa + 1, u) = 4 verify rows
        ai.logits = torch.cat([ai.logits[:, :2], ai.logits[:, 4:]], 1)
    h = dbv.Handle()
    try:
        dbv.sv_packed_anyorder_step(ai.logits.to(DEV), Kv, 4, ai.u.to(DEV), ai.win_pos.to(DEV),
                                    ai.order.to(DEV), ai.draft.to(DEV), ai.end_pos.to(DEV),
                                    handle=h)
        with pytest.raises(dbv.SVError) as e:
            h.sync_status()
        assert e.value.status == dbv.SV_ERR_DEVICE_BOUNDS
    finally:
        h.close()


def test_anyorder_full_size(dbv):
    """The any-order workload at full size (B = 256, 32 + 32 rows, V = 151936),
    against the oracle on the first 24 sequences."""
    c = datagen.CONFIGS["anyorder"]
    ai = datagen.anyorder_inputs(c["B"], c["K"], c["W"], c["V"], dtype="bf16", seed=c["seed"],
                                 device=DEV)
    out = dbv.sv_packed_anyorder_step(ai.logits, c["K"], c["W"], ai.u, ai.win_pos, ai.order,
                                      ai.draft, ai.end_pos)
    S = 24
    ref = oracle.packed_anyorder_step(np_logits(ai.logits[:S]), c["K"], c["W"], cpu(ai.u[:S]),
                                      cpu(ai.win_pos[:S]), cpu(ai.order[:S]), cpu(ai.draft[:S]),
                                      cpu(ai.end_pos[:S]))
    _compare_anyorder({k: v[:S] for k, v in out.items()}, ref, "bf16")
    assert ref["accept_len"].max() >= 2


# ------------------------------------------------------------------ Packed-SS

def _packed_both(dbv, pi, K, W, T, seed=7, it=3, eos=-1, rem=None, pos=None, handle=None):
    args = dict(T=T, seed=seed, it=it, eos_id=eos)
    out = dbv.sv_packed_step(_g(pi.logits), K, W, _g(pi.prev_draft), _g(pi.prev_len),
                             prev_q_at_draft=_g(pi.prev_q_at_draft),
                             prev_draft_logits=_g(pi.prev_draft_logits) if T > 0 else None,
                             prev_q_offset=_g(pi.prev_q_offset), pos_base=_g(pos),
                             remaining=_g(rem), handle=handle, **args)
    ref = oracle.packed_step(np_logits(pi.logits), K, W, cpu(pi.prev_draft), cpu(pi.prev_len),
                             cpu(pi.prev_q_at_draft) if T > 0 else None,
                             np_logits(pi.prev_draft_logits) if T > 0 else None,
                             cpu(pi.prev_q_offset), T=T, seed=seed, it=it,
                             pos_base=None if pos is None else cpu(pos), eos_id=eos,
                             remaining=None if rem is None else cpu(rem))
    return out, ref


def _compare_packed(out, ref, dtype):
    assert np.array_equal(cpu(out["flags"]), ref["flags"])
    keep = ref["flags"] == 0
    for k in ("accept_len", "commit_len", "committed", "next_draft", "next_len"):
        assert np.array_equal(cpu(out[k])[keep], ref[k][keep]), k
    assert_float_close(cpu(out["next_q_at_draft"])[keep], ref["next_q_at_draft"][keep],
                       RTOL[dtype], 0.0, "next_q_at_draft")
    assert_float_close(cpu(out["confidence"]), ref["confidence"], RTOL[dtype], 0.0, "confidence")


@pytest.mark.parametrize("T", [0.0, 1.0, 0.7])
@pytest.mark.parametrize("dtype,B,K,W,V", [("bf16", 6, 5, 5, 4104), ("f32", 4, 8, 6, 2048),
                                           ("bf16", 3, 32, 32, 1032), ("bf16", 4, 1, 3, 1024)])
def test_packed_parity(dbv, T, dtype, B, K, W, V):
    pi = datagen.packed_inputs(B, K, W, V, dtype=dtype, seed=K * 10 + W, T=T)
    pos = torch.arange(B, dtype=torch.int64) * 50 + 3
    out, ref = _packed_both(dbv, pi, K, W, T, pos=pos)
    _compare_packed(out, ref, dtype)
    # stopping by EOS and by the length cap
    eos = int(cpu(pi.prev_draft)[0, 0]) if K > 1 else 0
    rem = torch.randint(0, 4, (B,), dtype=torch.int32)
    out, ref = _packed_both(dbv, pi, K, W, T, eos=eos, rem=rem, pos=pos)
    _compare_packed(out, ref, dtype)


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_packed_fp64_path(dbv, T):
    pi = datagen.packed_inputs(6, 6, 6, 4104, dtype="bf16", seed=31, T=T)
    h = dbv.Handle()
    try:
        h.set_option(dbv.SV_OPT_FORCE_RESCUE, 1)
        out, ref = _packed_both(dbv, pi, 6, 6, T, handle=h)
        h.sync_status()
    finally:
        h.close()
    _compare_packed(out, ref, "bf16")


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_packed_full_size(dbv, T):
    """The Packed-SS workload at full size (B = 256, 32 + 32 rows, V = 151936 bf16),
    checked against the oracle on the first 24 sequences."""
    c = datagen.CONFIGS["packed"]
    B, K, W, V = c["B"], c["K"], c["W"], c["V"]
    pi = datagen.packed_inputs(B, K, W, V, dtype="bf16", seed=c["seed"], T=T, device=DEV)
    out = dbv.sv_packed_step(pi.logits, K, W, pi.prev_draft, pi.prev_len,
                             prev_q_at_draft=pi.prev_q_at_draft,
                             prev_draft_logits=pi.prev_draft_logits if T > 0 else None,
                             prev_q_offset=pi.prev_q_offset, T=T, seed=c["seed"], it=1)
    S = 24
    ref = oracle.packed_step(np_logits(pi.logits[:S]), K, W, cpu(pi.prev_draft[:S]),
                             cpu(pi.prev_len[:S]),
                             cpu(pi.prev_q_at_draft[:S]) if T > 0 else None,
                             np_logits(pi.prev_draft_logits[:S]) if T > 0 else None,
                             cpu(pi.prev_q_offset[:S]), T=T, seed=c["seed"], it=1)
    sub = {k: v[:S] for k, v in out.items()}
    _compare_packed(sub, ref, "bf16")


@pytest.mark.parametrize("B,W,V", [(152, 32, 8192), (160, 32, 8192), (8, 32, 151936)])
def test_packed_seed_spans(dbv, B, W, V):
    """The seed kernel splits the Gumbel-max rows' 256-id blocks, end to end,
    into one span per resident seed warp (4,864 on 152 SMs with four seed CTAs
    of eight warps each): 152 x 32 rows of 32 blocks give spans that are whole
    rows, 160 x 32 rows spans of 34 blocks that cut rows, and 8 x 32 rows of
    593 blocks spans of 32 blocks (a row in 19 or 20 pieces).  Every sequence
    is checked against the oracle."""
    K = 32
    pi = datagen.packed_inputs(B, K, W, V, dtype="bf16", seed=B + W, T=1.0)
    out, ref = _packed_both(dbv, pi, K, W, 1.0)
    _compare_packed(out, ref, "bf16")


# ------------------------------------------------------------------ errors

def test_invalid_arguments_raise(dbv):
    si = datagen.sample_inputs(2, 3, 1024, dtype="bf16", seed=1, device=DEV)
    with pytest.raises(dbv.SVError) as e:
        dbv.sv_verify_sample(si.target, si.draft, si.draft_ids, mode=1, lam=0.5)
    assert e.value.status == dbv.SV_ERR_INVALID_ARG
    with pytest.raises(dbv.SVError):
        dbv.sv_verify_sample(si.target, si.draft, si.draft_ids, mode=2, lam=1.5)
    bad = torch.zeros((2, 4, 1020), dtype=torch.bfloat16, device=DEV)  # V % 8 != 0
    with pytest.raises(dbv.SVError):
        dbv.sv_verify_greedy(bad, si.draft_ids)
    big = torch.zeros((1, 34, 64), dtype=torch.float32, device=DEV)  # K = 33 > 32
    with pytest.raises(dbv.SVError):
        dbv.sv_verify_greedy(big, torch.zeros((1, 33), dtype=torch.int32, device=DEV))


def test_out_of_range_ids_are_latched(dbv):
    si = datagen.sample_inputs(2, 3, 1024, dtype="bf16", seed=1, device=DEV)
    ids = si.draft_ids.clone()
    ids[1, 0] = 5000
    h = dbv.Handle()
    try:
        dbv.sv_verify_sample(si.target, si.draft, ids, handle=h)
        with pytest.raises(dbv.SVError) as e:
            h.sync_status()
        assert e.value.status == dbv.SV_ERR_DEVICE_BOUNDS
        # the handle stays usable afterwards
        out = dbv.sv_verify_sample(si.target, si.draft, si.draft_ids, handle=h)
        h.sync_status()
        ref = oracle.verify_sample(np_logits(si.target), np_logits(si.draft),
                                   cpu(si.draft_ids), want_tv=False)
        compare_sample(out, ref, "bf16", want_tv=False)
    finally:
        h.close()


def test_fp32_error_bounds_hold_on_device(dbv):
    """The bounds behind every certified fp32 decision hold on this GPU."""
    r = dbv.default_handle().selftest(seed=7, n=1 << 24)
    assert max(r[:3]) < 1.0, r
    assert r[3] == 0, r  # every fast skip gap equals the exact one
    assert r[4] == 0, r  # every G within its table bounds (ordinary and top ids)
