"""Failure paths on the GPU, made without faulting it.

- Bounded waits: a self-test kernel waits on an mbarrier that nothing
  arrives at and on a device word that nothing changes, with the kernels'
  own bounded-wait primitives and a small limit; both waits expire, the
  handle reports SV_ERR_TIMEOUT, and the next verify call on the same handle
  is exact again.
- Host fault injection: SV_FAULT_INJECT makes a verify call return an error
  status at its launch point; the binding raises it, nothing is enqueued,
  and the handle keeps working once the variable is cleared."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from gpu_util import DEV, compare_sample, cpu, np_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbv():
    import draft_block_verification_gb300 as m
    m.build()
    m.lib()
    oracle.build()
    return m


def _sample_case():
    si = datagen.sample_inputs(6, 5, 4104, dtype="bf16", seed=13, sigma=1.0, ragged=True)
    ref = oracle.verify_sample(np_logits(si.target), np_logits(si.draft), si.draft_ids.numpy(),
                               si.draft_len.numpy(), seed=9, want_tv=False)
    return si, ref


@pytest.mark.parametrize("limit", [0, 1, 1000])
def test_expired_waits_report_timeout_and_the_handle_recovers(dbv, limit):
    si, ref = _sample_case()
    h = dbv.Handle()
    try:
        h.wait_selftest(limit=limit)
        with pytest.raises(dbv.SVError) as e:
            h.sync_status()
        assert e.value.status == dbv.SV_ERR_TIMEOUT
        h.sync_status()  # the latched error was cleared with it
        out = dbv.sv_verify_sample(si.target.to(DEV), si.draft.to(DEV), si.draft_ids.to(DEV),
                                   si.draft_len.to(DEV), seed=9, handle=h)
        h.sync_status()
        compare_sample(out, ref, "bf16", want_tv=False)
    finally:
        h.close()


def test_wait_selftest_rejects_bad_limits(dbv):
    h = dbv.Handle()
    try:
        for bad in (-1, 1 << 25):
            with pytest.raises(dbv.SVError) as e:
                h.wait_selftest(limit=bad)
            assert e.value.status == dbv.SV_ERR_INVALID_ARG
    finally:
        h.close()


@pytest.mark.parametrize("call,code", [("sv_verify_sample", 2), ("sv_verify_sample", 3),
                                       ("sv_packed_step", 2), ("sv_verify_tree", 3),
                                       ("sv_verify_greedy", 2), ("sv_verify_greedy_static", 3)])
def test_injected_launch_failures(dbv, monkeypatch, call, code):
    si, ref = _sample_case()
    tgt, drf, ids, dl = (t.to(DEV) for t in (si.target, si.draft, si.draft_ids, si.draft_len))
    h = dbv.Handle()
    try:
        monkeypatch.setenv("SV_FAULT_INJECT", "%s:%d" % (call, code))
        with pytest.raises(dbv.SVError) as e:
            if call == "sv_verify_sample":
                dbv.sv_verify_sample(tgt, drf, ids, dl, seed=9, handle=h)
            elif call == "sv_verify_greedy":
                dbv.sv_verify_greedy(tgt, ids, dl, handle=h)
            elif call == "sv_verify_greedy_static":
                dbv.sv_verify_greedy_static(tgt, ids, dl)
            elif call == "sv_verify_tree":
                par = torch.full((6, 4), -1, dtype=torch.int32, device=DEV)
                dbv.sv_verify_tree(tgt[:, :4].contiguous(), par, par + 1, par + 1, T=1.0,
                                   handle=h)
            else:
                pi = datagen.packed_inputs(2, 3, 3, 1024, dtype="bf16", seed=2, T=0.0,
                                           device=DEV)
                dbv.sv_packed_step(pi.logits, 3, 3, pi.prev_draft, pi.prev_len, T=0.0,
                                   handle=h)
        assert e.value.status == code
        h.sync_status()  # nothing was enqueued, nothing latched
        # other calls are unaffected by the injection
        if call != "sv_verify_sample":
            out = dbv.sv_verify_sample(tgt, drf, ids, dl, seed=9, handle=h)
            h.sync_status()
            compare_sample(out, ref, "bf16", want_tv=False)
        monkeypatch.delenv("SV_FAULT_INJECT")
        out = dbv.sv_verify_sample(tgt, drf, ids, dl, seed=9, handle=h)
        h.sync_status()
        compare_sample(out, ref, "bf16", want_tv=False)
    finally:
        h.close()
