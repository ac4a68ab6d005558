"""GPU parity of the Packed-SS step with top-k truncated distributions
(sv_packed_topk_step) against the oracle: decisions, committed blocks, next
drafts and the stored lists bit-exact wherever neither side flagged a
decision; probabilities within fp32 rounding.  Inputs are two consecutive
calls: the first (no previous draft) on the previous rows, whose lists and
drafts, computed by the oracle, become the second call's state."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from gpu_util import DEV, assert_float_close, cpu, np_logits

pytestmark = pytest.mark.gpu

OUT_KEYS = ("accept_len", "commit_len", "committed", "next_draft", "next_len")
QTOL = 4e-6


@pytest.fixture(scope="module")
def dbv():
    import draft_block_verification_gb300 as m
    m.build()
    m.lib()
    oracle.build()
    return m


def _first_call(logits_np, K, W, kp, kq, T, seed, it):
    B = logits_np.shape[0]
    return oracle.packed_topk_step(logits_np, K, W, kp, kq, np.zeros((B, K - 1), np.int32),
                                   np.zeros(B, np.int32), np.zeros((B, W, kq), np.int32),
                                   np.zeros((B, W, kq), np.float32), np.zeros(B, np.int32), T,
                                   seed=seed, it=it)


def _gpu(dbv, logits, K, W, kp, kq, st, T, seed, it, **kw):
    t = {k: torch.as_tensor(v).to(DEV) for k, v in st.items()}
    return dbv.sv_packed_topk_step(logits, K, W, kp, kq, t["prev_draft"], t["prev_len"],
                                   t["prev_q_ids"], t["prev_q_probs"], t["prev_q_offset"], T=T,
                                   seed=seed, it=it, **kw)


def _compare(out, ref, kq):
    fg, fr = cpu(out["flags"]), ref["flags"]
    assert np.array_equal(fg, fr), "flag counts differ"
    keep = fr == 0
    for k in OUT_KEYS:
        assert np.array_equal(cpu(out[k])[keep], ref[k][keep]), k
    assert np.array_equal(cpu(out["q_ids"]), ref["q_ids"])
    # the stored probabilities are fp32 outputs whose terms are taken in fp32
    # (an expf of an argument rounded to fp32: under 2^-24 |arg| + 2 ulp)
    assert_float_close(cpu(out["q_probs"]), ref["q_probs"], QTOL, 1e-12, "q_probs")
    assert_float_close(cpu(out["next_q_at_draft"])[keep], ref["next_q_at_draft"][keep], QTOL,
                       1e-12, "next_q_at_draft")
    return int(keep.sum())


def _two_calls(B, K, W, V, kp, kq, T, dtype, seed, sigma=0.3):
    ti = datagen.packed_topk_inputs(B, K, W, V, dtype=dtype, seed=seed, sigma=sigma)
    prev = _first_call(np_logits(ti.prev_logits), K, W, kp, kq, T, seed, 1)
    a_prev = np.maximum(ti.a_prev.numpy(), prev["commit_len"])
    st = datagen.packed_state_from(prev["next_draft"], prev["commit_len"], prev["q_ids"],
                                   prev["q_probs"].astype(np.float32), a_prev, K, W)
    return ti, prev, st


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("kp,kq,T", [(1, 1, 1.0), (5, 3, 0.7), (20, 20, 1.0), (64, 64, 1.0),
                                     (3, 17, 1.3)])
def test_topk_parity(dbv, dtype, kp, kq, T):
    B, K, W, V, seed = 20, 6, 7, 4104, 31 + kp + kq
    ti, prev, st = _two_calls(B, K, W, V, kp, kq, T, dtype, seed)
    # the first call (no previous draft): bonus tokens and lists
    zst = dict(prev_draft=np.zeros((B, K - 1), np.int32), prev_len=np.zeros(B, np.int32),
               prev_q_offset=np.zeros(B, np.int32), prev_q_ids=np.zeros((B, W, kq), np.int32),
               prev_q_probs=np.zeros((B, W, kq), np.float32))
    out = _gpu(dbv, ti.prev_logits.to(DEV), K, W, kp, kq, zst, T, seed, 1)
    _compare(out, prev, kq)
    # the second call verifies the first call's drafts against its lists
    ref = oracle.packed_topk_step(np_logits(ti.logits), K, W, kp, kq, seed=seed, it=2, T=T, **st)
    out = _gpu(dbv, ti.logits.to(DEV), K, W, kp, kq, st, T, seed, 2)
    assert _compare(out, ref, kq) >= B - 1
    if kp > 1:
        assert ref["accept_len"].max() >= 1  # some drafts are accepted
        assert (ref["accept_len"] < st["prev_len"]).any()  # and some rejected


def test_topk_ties_and_small_vocab(dbv):
    """Rows with many equal logits (integers) and k = V: the selection's
    tie rule (lower id first) decides the lists."""
    B, K, W, V, k, T = 6, 3, 4, 64, 64, 1.0
    rng = np.random.default_rng(4)
    prev = torch.tensor(rng.integers(-2, 3, (B, K + W, V)).astype(np.float32))
    cur = torch.tensor(rng.integers(-2, 3, (B, K + W, V)).astype(np.float32))
    pr = _first_call(prev.numpy(), K, W, k, 9, T, 3, 0)
    st = datagen.packed_state_from(pr["next_draft"], pr["commit_len"], pr["q_ids"],
                                   pr["q_probs"].astype(np.float32),
                                   np.maximum(pr["commit_len"], 2), K, W)
    for kp, kq, logits in ((k, 9, prev), (7, 9, cur)):
        s = st if logits is cur else dict(
            prev_draft=np.zeros((B, K - 1), np.int32), prev_len=np.zeros(B, np.int32),
            prev_q_offset=np.zeros(B, np.int32), prev_q_ids=np.zeros((B, W, kq), np.int32),
            prev_q_probs=np.zeros((B, W, kq), np.float32))
        ref = oracle.packed_topk_step(logits.numpy(), K, W, kp, kq, T=T, seed=3, it=0, **s)
        out = _gpu(dbv, logits.to(DEV), K, W, kp, kq, s, T, 3, 0)
        _compare(out, ref, kq)


def test_topk_clustered_row_takes_the_rescan(dbv):
    """A row whose largest logits sit in a few 16-byte vectors (increasing
    logits over the vocabulary) leaves some threads of the selection with more
    than four of the top k: the rescan path must still give the exact list."""
    B, K, W, V, k, T = 2, 2, 2, 8192, 64, 1.0
    base = np.linspace(-3, 3, V).astype(np.float32)
    logits = np.broadcast_to(base, (B, K + W, V)).copy()
    logits[1] = logits[1][:, ::-1]
    zst = dict(prev_draft=np.zeros((B, K - 1), np.int32), prev_len=np.zeros(B, np.int32),
               prev_q_offset=np.zeros(B, np.int32), prev_q_ids=np.zeros((B, W, k), np.int32),
               prev_q_probs=np.zeros((B, W, k), np.float32))
    ref = oracle.packed_topk_step(logits, K, W, k, k, T=T, seed=5, **zst)
    out = _gpu(dbv, torch.tensor(logits).to(DEV), K, W, k, k, zst, T, 5, 0)
    _compare(out, ref, k)


def test_topk_full_size(dbv):
    """The bench workload: B = 256, K = W = 32, V = 151,936 bf16, k = 20."""
    c = datagen.CONFIGS["packed_topk"]
    B, K, W, V, kp, kq, T, seed = (c[x] for x in ("B", "K", "W", "V", "kp", "kq", "T", "seed"))
    ti, prev, st = _two_calls(B, K, W, V, kp, kq, T, c["dtype"], seed)
    ref = oracle.packed_topk_step(np_logits(ti.logits), K, W, kp, kq, seed=seed, it=2, T=T, **st)
    out = _gpu(dbv, ti.logits.to(DEV), K, W, kp, kq, st, T, seed, 2)
    assert _compare(out, ref, kq) >= B - 2
    assert ref["accept_len"].mean() > 1.0


def test_topk_draft_missing_from_its_list_latches(dbv):
    B, K, W, V, k = 2, 3, 3, 64, 4
    logits = torch.randn(B, K + W, V).to(DEV)
    st = dict(prev_draft=np.array([[63, 0], [63, 0]], np.int32), prev_len=np.ones(B, np.int32),
              prev_q_offset=np.zeros(B, np.int32),
              prev_q_ids=np.tile(np.arange(k, dtype=np.int32), (B, W, 1)),
              prev_q_probs=np.full((B, W, k), 0.25, np.float32))
    h = dbv.Handle()
    try:
        _gpu(dbv, logits, K, W, k, k, st, 1.0, 0, 0, handle=h)
        with pytest.raises(dbv.SVError) as e:
            h.sync_status()
        assert e.value.status == dbv.SV_ERR_DEVICE_BOUNDS
    finally:
        h.close()


def test_topk_rejects_bad_arguments(dbv):
    logits = torch.randn(1, 4, 64).to(DEV)
    st = dict(prev_draft=np.zeros((1, 1), np.int32), prev_len=np.zeros(1, np.int32),
              prev_q_offset=np.zeros(1, np.int32), prev_q_ids=np.zeros((1, 2, 4), np.int32),
              prev_q_probs=np.zeros((1, 2, 4), np.float32))
    for kp, kq, T in ((0, 4, 1.0), (65, 4, 1.0), (4, 4, 0.0)):
        s = dict(st)
        with pytest.raises(dbv.SVError) as e:
            _gpu(dbv, logits, 2, 2, kp, 4, s, T, 0, 0)
        assert e.value.status == dbv.SV_ERR_INVALID_ARG
