"""sv_verify_greedy_static: the allocation-free greedy call gives the same
results as sv_verify_greedy, call after call, allocates no device memory,
reports device-side errors through its status word and rejects shapes beyond
its fixed scratch.  Kept in a file of its own, collected last, so that it runs
both alone and after every other GPU test in the same process."""
import pytest
import torch

import datagen

pytestmark = pytest.mark.gpu

SV_ERR_UNSUPPORTED = 5
SV_ERR_DEVICE_BOUNDS = 6


@pytest.fixture(scope="module")
def dbv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import draft_block_verification_gb300 as m
    return m


def _case(B, K, V, dtype, seed, ragged):
    dev = torch.device("cuda", 0)
    gi = datagen.greedy_inputs(B, K, V, dtype=dtype, seed=seed, ragged=ragged)
    return gi.target.to(dev), gi.draft_ids.to(dev), gi.draft_len.to(dev)


def test_matches_handle_path_on_consecutive_calls(dbv):
    cases = [_case(5, 8, 32000, "bf16", 11, True), _case(8, 16, 151936, "bf16", 12, False),
             _case(3, 5, 4104, "f32", 13, True)]
    for target, ids, dl in cases:
        ref_acc, ref_nxt = dbv.sv_verify_greedy(target, ids, dl)
        acc, nxt, st = dbv.sv_verify_greedy_static(target, ids, dl)
        torch.cuda.synchronize()
        assert int(st[0]) == 0
        assert torch.equal(acc, ref_acc)
        assert torch.equal(nxt, ref_nxt)


def test_allocates_no_device_memory(dbv):
    target, ids, dl = _case(16, 8, 151936, "bf16", 21, True)
    acc = torch.empty(16, dtype=torch.int32, device=target.device)
    nxt = torch.empty_like(acc)
    st = torch.empty(1, dtype=torch.int32, device=target.device)
    dbv.sv_verify_greedy_static(target, ids, dl, accept_len=acc, next_token=nxt, status=st)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        dbv.sv_verify_greedy_static(target, ids, dl, accept_len=acc, next_token=nxt, status=st)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    ref_acc, ref_nxt = dbv.sv_verify_greedy(target, ids, dl)
    assert torch.equal(acc, ref_acc) and torch.equal(nxt, ref_nxt) and int(st[0]) == 0


def test_status_reports_device_errors_and_next_call_starts_clean(dbv):
    target, ids, dl = _case(4, 6, 4104, "bf16", 31, False)
    bad = dl.clone()
    bad[2] = 99  # beyond K: latched on the device, the length is clamped
    _, _, st = dbv.sv_verify_greedy_static(target, ids, bad)
    torch.cuda.synchronize()
    assert int(st[0]) == SV_ERR_DEVICE_BOUNDS
    acc, nxt, st = dbv.sv_verify_greedy_static(target, ids, dl)
    ref_acc, ref_nxt = dbv.sv_verify_greedy(target, ids, dl)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    assert torch.equal(acc, ref_acc) and torch.equal(nxt, ref_nxt)


@pytest.mark.parametrize("B,K,V,dtype,ragged", [(4096, 7, 64, "bf16", True),
                                                 (4096, 7, 1032, "f32", False),
                                                 (300, 0, 4104, "bf16", False)])
def test_capacity_limit_and_no_draft_tokens(dbv, B, K, V, dtype, ragged):
    """At the limit (B = 4096 and B * (K + 1) = 32768 rows: one part per row,
    every record and counter of the scratch in use) and with no draft tokens,
    the results equal the handle path's on two calls in a row."""
    target, ids, dl = _case(B, K, V, dtype, B + K, ragged)
    ref_acc, ref_nxt = dbv.sv_verify_greedy(target, ids, dl)
    for _ in range(2):
        acc, nxt, st = dbv.sv_verify_greedy_static(target, ids, dl)
        torch.cuda.synchronize()
        assert int(st[0]) == 0
        assert torch.equal(acc, ref_acc) and torch.equal(nxt, ref_nxt)


def test_empty_batch(dbv):
    dev = torch.device("cuda", 0)
    target = torch.zeros((0, 4, 64), dtype=torch.bfloat16, device=dev)
    ids = torch.zeros((0, 3), dtype=torch.int32, device=dev)
    acc, nxt, st = dbv.sv_verify_greedy_static(target, ids)
    torch.cuda.synchronize()
    assert acc.numel() == 0 and nxt.numel() == 0 and int(st[0]) == 0


@pytest.mark.parametrize("B,K", [(4097, 0), (1025, 31)])
def test_rejects_shapes_beyond_the_scratch(dbv, B, K):
    dev = torch.device("cuda", 0)
    target = torch.zeros((B, K + 1, 8), dtype=torch.bfloat16, device=dev)
    ids = torch.zeros((B, K), dtype=torch.int32, device=dev)
    with pytest.raises(dbv.SVError) as e:
        dbv.sv_verify_greedy_static(target, ids)
    assert e.value.status == SV_ERR_UNSUPPORTED
