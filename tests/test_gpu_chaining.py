"""GPU parity of calls that follow one another on a stream with no host
synchronisation in between, and of batches larger than the GPU's SM count.

The library's kernels are chained by programmatic dependent launch: each may be
scheduled while the previous kernel of the stream drains, and waits for it on
the device before it touches global memory.  These tests enqueue calls of
every kind back to back (sharing one handle, whose workspace counters every
call must leave at zero) and check every result against the oracle only at
the end.  The large batches make the residual kernel's CTAs take several
sequences each and leave many decision steps for the end of the streaming
pass."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from gpu_util import DEV, cpu, compare_sample, craft_tree_tokens, np_logits

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


def _sample_ref(si, T, mode, lam, seed, pos=None):
    return oracle.verify_sample(np_logits(si.target), np_logits(si.draft), si.draft_ids.numpy(),
                                si.draft_len.numpy(), T_p=T, T_q=T, mode=mode, lam=lam,
                                seed=seed, pos_base=None if pos is None else pos.numpy())


def test_back_to_back_calls_without_sync(dbv):
    h = dbv.Handle()
    try:
        # 1. sampling (lossless), 2. tree at T = 1, 3. Packed-SS at T = 1,
        # 4. greedy, 5. sampling again with other shapes and a lenient rule
        s1 = datagen.sample_inputs(8, 6, 8200, dtype="bf16", seed=11, sigma=0.5)
        ti = datagen.tree_inputs(3, 24, 4096, dtype="bf16", seed=12, L=16, max_depth=8)
        tok = craft_tree_tokens(np_logits(ti.node_logits), ti.node_pos.numpy(), 1.0, 5,
                                np.random.default_rng(3))
        pk = datagen.packed_inputs(4, 6, 6, 4104, dtype="bf16", seed=13, T=1.0)
        gi = datagen.greedy_inputs(3, 5, 4104, dtype="f32", seed=14, ragged=True)
        s2 = datagen.sample_inputs(5, 9, 12288, dtype="bf16", seed=15, sigma=1.0, T=0.7,
                                   ragged=True)
        dev = [_g(t) for t in (s1.target, s1.draft, s1.draft_ids, ti.node_logits, ti.parent,
                               ti.node_pos, torch.from_numpy(tok), pk.logits, pk.prev_draft,
                               pk.prev_len, pk.prev_q_at_draft, pk.prev_draft_logits,
                               pk.prev_q_offset, gi.target, gi.draft_ids, gi.draft_len,
                               s2.target, s2.draft, s2.draft_ids, s2.draft_len)]
        torch.cuda.synchronize()
        (t1, d1, i1, tl, tp, tn, tt, pl, pd, pn, pq, pdl, po, gt, gd, gl, t2, d2, i2,
         l2) = dev
        o1 = dbv.sv_verify_sample(t1, d1, i1, T_p=1.0, T_q=1.0, seed=41, handle=h)
        o2 = dbv.sv_verify_tree(tl, tp, tn, tt, T=1.0, seed=5, max_depth=8, handle=h)
        o3 = dbv.sv_packed_step(pl, 6, 6, pd, pn, prev_q_at_draft=pq, prev_draft_logits=pdl,
                                prev_q_offset=po, T=1.0, seed=7, it=2, handle=h)
        a4, n4 = dbv.sv_verify_greedy(gt, gd, gl, handle=h)
        o5 = dbv.sv_verify_sample(t2, d2, i2, l2, T_p=0.7, T_q=0.7, mode=dbv.SV_LENIENT_RATIO,
                                  lam=4.0, seed=42, want_tv=True, handle=h)
        h.sync_status()
    finally:
        h.close()

    compare_sample(o1, _sample_ref(s1, 1.0, 0, 1.0, 41), "bf16")
    r2 = oracle.verify_tree(np_logits(ti.node_logits), ti.parent.numpy(), ti.node_pos.numpy(),
                            tok, T=1.0, seed=5, max_depth=8)
    assert np.array_equal(cpu(o2["flags"]), r2["flags"])
    keep = r2["flags"] == 0
    for k in ("path_len", "commit_count", "path_nodes", "match"):
        assert np.array_equal(cpu(o2[k])[keep], r2[k][keep]), k
    r3 = oracle.packed_step(np_logits(pk.logits), 6, 6, cpu(pk.prev_draft), cpu(pk.prev_len),
                            cpu(pk.prev_q_at_draft), np_logits(pk.prev_draft_logits),
                            cpu(pk.prev_q_offset), T=1.0, seed=7, it=2)
    assert np.array_equal(cpu(o3["flags"]), r3["flags"])
    keep = r3["flags"] == 0
    for k in ("accept_len", "commit_len", "committed", "next_draft", "next_len"):
        assert np.array_equal(cpu(o3[k])[keep], r3[k][keep]), k
    r4 = oracle.verify_greedy(np_logits(gi.target), gi.draft_ids.numpy(), gi.draft_len.numpy())
    assert np.array_equal(cpu(a4), r4["accept_len"])
    assert np.array_equal(cpu(n4), r4["next_token"])
    compare_sample(o5, _sample_ref(s2, 0.7, dbv.SV_LENIENT_RATIO, 4.0, 42), "bf16")


@pytest.mark.parametrize("B,K,V,mode,lam", [(200, 3, 1032, 0, 1.0), (600, 2, 520, 1, 2.0)])
def test_sample_more_sequences_than_sms(dbv, B, K, V, mode, lam):
    """More sequences than SMs: residual CTAs loop over several rejecting
    sequences, and many decision steps fall to the end of the pass."""
    si = datagen.sample_inputs(B, K, V, dtype="bf16", seed=B + K, sigma=1.0)
    pos = torch.arange(B, dtype=torch.int64) * 3 + 1
    out = dbv.sv_verify_sample(_g(si.target), _g(si.draft), _g(si.draft_ids), T_p=1.0,
                               T_q=1.0, mode=mode, lam=lam, seed=17, pos_base=_g(pos))
    ref = _sample_ref(si, 1.0, mode, lam, 17, pos)
    compare_sample(out, ref, "bf16")
    dbv.default_handle().sync_status()
    assert (ref["accept_len"] < K).sum() > 64  # the residual pass has real work


def test_repeated_calls_same_handle(dbv):
    """The same call ten times on one handle without synchronising: every
    result equals the first (counters return to zero between calls)."""
    si = datagen.sample_inputs(16, 8, 16392, dtype="bf16", seed=77, sigma=0.5, device=DEV)
    h = dbv.Handle()
    try:
        outs = [dbv.sv_verify_sample(si.target, si.draft, si.draft_ids, T_p=1.0, T_q=1.0,
                                     seed=3, handle=h) for _ in range(10)]
        h.sync_status()
    finally:
        h.close()
    for o in outs[1:]:
        for k in ("accept_len", "next_token", "flags"):
            assert np.array_equal(cpu(o[k]), cpu(outs[0][k])), k
