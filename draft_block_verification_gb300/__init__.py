"""draft_block_verification_gb300: draft-block verification on GB300 (sm_103a).

A thin ctypes binding over the C ABI of ``libsv.so`` (declared in
``include/sv.h``).  Each function has the C name, takes torch CUDA tensors,
marshals pointers, sizes and the current CUDA stream, and raises ``SVError``
on any status other than SV_OK.  Every step of the computation runs in the
library's kernels; there is no other code path.  The library must have been
built (``draft_block_verification_gb300._build.build()``); importing the
functions when it is missing raises immediately.
"""
from __future__ import annotations

import atexit
import ctypes as C
import os
import sys
import threading

import torch

from ._build import LIBPATH, build  # noqa: F401  (build is part of the API)

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_CUDA, SV_ERR_OOM = 0, 1, 2, 3
SV_ERR_TIMEOUT, SV_ERR_UNSUPPORTED, SV_ERR_DEVICE_BOUNDS = 4, 5, 6
SV_F32, SV_BF16 = 0, 1
SV_LOSSLESS, SV_LENIENT_RATIO, SV_LENIENT_LINEAR, SV_LENIENT_CACTUS = 0, 1, 2, 3
SV_OPT_FORCE_RESCUE, SV_OPT_TIMING_EVENTS = 1, 2

_lib = None
_lock = threading.Lock()
_handles = {}


class SVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


def lib():
    """The loaded libsv.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBPATH):
            raise RuntimeError("libsv.so is not built: run draft_block_verification_gb300."
                               "_build.build() (nvcc with sm_103a support)")
        L = C.CDLL(LIBPATH)
        vp, i32, i64, u64, f32 = C.c_void_p, C.c_int, C.c_int64, C.c_uint64, C.c_float
        L.sv_status_string.restype, L.sv_status_string.argtypes = C.c_char_p, [i32]
        L.sv_create.restype, L.sv_create.argtypes = i32, [C.POINTER(vp)]
        L.sv_destroy.restype, L.sv_destroy.argtypes = i32, [vp]
        L.sv_sync_status.restype, L.sv_sync_status.argtypes = i32, [vp, vp]
        L.sv_rescue_count.restype = i32
        L.sv_rescue_count.argtypes = [vp, vp, C.POINTER(C.c_int64)]
        L.sv_set_option.restype, L.sv_set_option.argtypes = i32, [vp, i32, i64]
        L.sv_selftest.restype = i32
        L.sv_selftest.argtypes = [vp, u64, i64, C.POINTER(C.c_double), vp]
        L.sv_wait_selftest.restype, L.sv_wait_selftest.argtypes = i32, [vp, i64, vp]
        L.sv_verify_greedy.restype = i32
        L.sv_verify_greedy.argtypes = [vp, vp, i32, i64, i32, i32, i32, vp, vp, vp, vp, vp]
        L.sv_verify_greedy_static.restype = i32
        L.sv_verify_greedy_static.argtypes = [vp, i32, i64, i32, i32, i32, vp, vp, vp, vp, vp,
                                              vp]
        L.sv_verify_sample.restype = i32
        L.sv_verify_sample.argtypes = [vp, vp, vp, i32, i64, i32, i32, i32, vp, vp, f32, f32,
                                       i32, f32, u64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.sv_verify_tree.restype = i32
        L.sv_verify_tree.argtypes = [vp, vp, i32, i64, i32, i32, i32, vp, vp, vp, f32, u64, vp,
                                     vp, vp, i32, vp, vp, vp, vp]
        L.sv_verify_spot.restype = i32
        L.sv_verify_spot.argtypes = [vp, vp, i32, i64, i32, i32, i32, i32, vp, vp, vp, vp, f32,
                                     u64, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.sv_packed_anyorder_step.restype = i32
        L.sv_packed_anyorder_step.argtypes = [vp, vp, i32, i64, i32, i32, i32, i32, vp, vp, vp,
                                              vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.sv_packed_step.restype = i32
        L.sv_packed_step.argtypes = [vp, vp, i32, i64, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                     f32, u64, u64, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                     vp]
        L.sv_packed_topk_step.restype = i32
        L.sv_packed_topk_step.argtypes = [vp, vp, i32, i64, i32, i32, i32, i32, i32, i32, vp, vp,
                                          vp, vp, vp, f32, u64, u64, vp, i32, vp, vp, vp, vp, vp,
                                          vp, vp, vp, vp, vp, vp]
        _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().sv_status_string(int(s)).decode()


def _check(s: int, where: str):
    if s != SV_OK:
        raise SVError(s, where)


class Handle:
    """An sv_handle bound to one CUDA device."""

    def __init__(self, device=None):
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None
                                   else torch.device(device).index or 0)
        with torch.cuda.device(self.device):
            h = C.c_void_p()
            _check(lib().sv_create(C.byref(h)), "sv_create")
        self.ptr = h

    def close(self):
        if self.ptr:
            lib().sv_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        # At interpreter shutdown the CUDA runtime may already be gone; the
        # process exit releases the device memory then.
        if sys.is_finalizing():
            return
        try:
            self.close()
        except Exception:
            pass

    def sync_status(self, stream=None):
        """Synchronise and raise the first device-side error latched."""
        _check(lib().sv_sync_status(self.ptr, _stream(stream, self.device)), "device")

    def rescue_count(self, stream=None) -> int:
        c = C.c_int64()
        _check(lib().sv_rescue_count(self.ptr, _stream(stream, self.device), C.byref(c)),
               "sv_rescue_count")
        return int(c.value)

    def selftest(self, seed: int = 1, n: int = 1 << 22, stream=None):
        """Ratios of the measured fp32 errors to the bounds the kernels assume,
        the count of skip gaps whose fast evaluation is not exact, and the
        count of ids outside their Gumbel bound table entries."""
        r = (C.c_double * 5)()
        _check(lib().sv_selftest(self.ptr, int(seed), int(n), r, _stream(stream, self.device)),
               "sv_selftest")
        return list(r)

    def wait_selftest(self, limit: int = 1000, stream=None):
        """Enqueue the self-test whose bounded waits run out: the next
        sync_status raises SVError with SV_ERR_TIMEOUT."""
        _check(lib().sv_wait_selftest(self.ptr, int(limit), _stream(stream, self.device)),
               "sv_wait_selftest")

    def set_option(self, opt: int, value: int):
        _check(lib().sv_set_option(self.ptr, int(opt), int(value)), "sv_set_option")


@atexit.register
def _close_default_handles():
    with _lock:
        for h in _handles.values():
            try:
                h.close()
            except Exception:
                pass
        _handles.clear()


def default_handle(device=None) -> Handle:
    dev = torch.cuda.current_device() if device is None else torch.device(device).index or 0
    with _lock:
        if dev not in _handles:
            _handles[dev] = Handle(dev)
        return _handles[dev]


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _rows(t, name):
    """(dtype code, row stride in elements) of a [..., rows, V] logit tensor."""
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype == torch.bfloat16:
        code = SV_BF16
    elif t.dtype == torch.float32:
        code = SV_F32
    else:
        raise ValueError("%s must be bfloat16 or float32" % name)
    if t.stride(-1) != 1:
        raise ValueError("%s: the vocabulary dimension must be contiguous" % name)
    rs = t.stride(-2) if t.dim() >= 2 else t.shape[-1]
    for d in range(t.dim() - 2):
        if t.stride(d) != t.shape[d + 1] * t.stride(d + 1):
            raise ValueError("%s: rows must be evenly strided" % name)
    return code, rs


def _i32(t, shape, name, dev):
    if t is None:
        return None
    if t.dtype != torch.int32 or not t.is_cuda or t.device != dev or not t.is_contiguous():
        raise ValueError("%s must be a contiguous int32 tensor on %s" % (name, dev))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s" % (name, tuple(shape)))
    return t


def _out(t, shape, dtype, dev):
    return torch.empty(shape, dtype=dtype, device=dev) if t is None else t


def sv_verify_greedy(target, draft_ids, draft_len=None, *, handle=None, stream=None,
                     accept_len=None, next_token=None):
    """Greedy verification; target [B, K+1, V]; returns (accept_len, next_token)."""
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    code, rs = _rows(target, "target")
    h = handle or default_handle(dev)
    ids = _i32(draft_ids, (B, K), "draft_ids", dev)
    dl = _i32(draft_len, (B,), "draft_len", dev)
    acc = _out(accept_len, (B,), torch.int32, dev)
    nxt = _out(next_token, (B,), torch.int32, dev)
    _check(lib().sv_verify_greedy(h.ptr, _p(target), code, rs, B, K, V, _p(ids), _p(dl),
                                  _p(acc), _p(nxt), _stream(stream, dev)), "sv_verify_greedy")
    return acc, nxt


def sv_verify_greedy_static(target, draft_ids, draft_len=None, *, stream=None, accept_len=None,
                            next_token=None, status=None):
    """Greedy verification with the library's fixed scratch (no device
    allocation by the library; see sv.h).  Returns (accept_len, next_token,
    status); status[0] holds the first device-side error of the call, 0 if
    none.  Pass preallocated outputs to keep the call free of allocations on
    the Python side as well."""
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    code, rs = _rows(target, "target")
    ids = _i32(draft_ids, (B, K), "draft_ids", dev)
    dl = _i32(draft_len, (B,), "draft_len", dev)
    acc = _out(accept_len, (B,), torch.int32, dev)
    nxt = _out(next_token, (B,), torch.int32, dev)
    st = _out(status, (1,), torch.int32, dev)
    _check(lib().sv_verify_greedy_static(_p(target), code, rs, B, K, V, _p(ids), _p(dl), _p(acc),
                                         _p(nxt), _p(st), _stream(stream, dev)),
           "sv_verify_greedy_static")
    return acc, nxt, st


def sv_verify_sample(target, draft, draft_ids, draft_len=None, *, T_p=1.0, T_q=1.0,
                     mode=SV_LOSSLESS, lam=1.0, seed=0, pos_base=None, want_rows=True,
                     want_tv=False, handle=None, stream=None):
    """Lossless / lenient speculative sampling; target [B, K+1, V], draft [B, K, V].
    Returns a dict of output tensors (see sv.h)."""
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    code, rs = _rows(target, "target")
    if K > 0:
        code2, rs2 = _rows(draft, "draft")
        if code2 != code or rs2 != rs or tuple(draft.shape) != (B, K, V):
            raise ValueError("draft must be [B, K, V] with the target's dtype and row stride")
    h = handle or default_handle(dev)
    ids = _i32(draft_ids, (B, K), "draft_ids", dev)
    dl = _i32(draft_len, (B,), "draft_len", dev)
    if pos_base is not None and (pos_base.dtype != torch.int64 or not pos_base.is_cuda):
        raise ValueError("pos_base must be an int64 CUDA tensor")
    f = lambda *s: torch.empty(s, dtype=torch.float32, device=dev)
    out = {"accept_len": torch.empty(B, dtype=torch.int32, device=dev),
           "next_token": torch.empty(B, dtype=torch.int32, device=dev),
           "flags": torch.empty(B, dtype=torch.int32, device=dev)}
    if want_rows:
        out.update(p_at_draft=f(B, K), q_at_draft=f(B, K), lse_p=f(B, K + 1), lse_q=f(B, K))
    if want_tv:
        out["tv"] = f(B, K)
    g = out.get
    _check(lib().sv_verify_sample(
        h.ptr, _p(target), _p(draft) if K > 0 else None, code, rs, B, K, V, _p(ids), _p(dl),
        float(T_p), float(T_q), int(mode), float(lam), int(seed) & (2**64 - 1), _p(pos_base),
        _p(out["accept_len"]), _p(out["next_token"]), _p(g("p_at_draft")), _p(g("q_at_draft")),
        _p(g("lse_p")), _p(g("lse_q")), _p(g("tv")), _p(out["flags"]), _stream(stream, dev)),
        "sv_verify_sample")
    return out


def sv_verify_tree(node_logits, parent, node_pos, node_tok, *, T=0.0, seed=0, pos_base=None,
                   max_depth=None, handle=None, stream=None):
    """Coupled-noise tree verification; node_logits [B, N, V]."""
    B, N, V = node_logits.shape
    dev = node_logits.device
    code, rs = _rows(node_logits, "node_logits")
    h = handle or default_handle(dev)
    par = _i32(parent, (B, N), "parent", dev)
    pos = _i32(node_pos, (B, N), "node_pos", dev)
    tok = _i32(node_tok, (B, N), "node_tok", dev)
    md = N if max_depth is None else int(max_depth)
    out = {"path_len": torch.empty(B, dtype=torch.int32, device=dev),
           "path_nodes": torch.empty((B, md), dtype=torch.int32, device=dev),
           "commit_count": torch.empty(B, dtype=torch.int32, device=dev),
           "match": torch.empty((B, N), dtype=torch.uint8, device=dev),
           "flags": torch.empty(B, dtype=torch.int32, device=dev)}
    _check(lib().sv_verify_tree(
        h.ptr, _p(node_logits), code, rs, B, N, V, _p(par), _p(pos), _p(tok), float(T),
        int(seed) & (2**64 - 1), _p(pos_base), _p(out["path_len"]), _p(out["path_nodes"]), md,
        _p(out["commit_count"]), _p(out["match"]), _p(out["flags"]), _stream(stream, dev)),
        "sv_verify_tree")
    return out


def sv_verify_spot(state_logits, parent, node_pos, node_tok, root_mask, *, T=0.0, seed=0,
                   pos_base=None, max_depth=None, handle=None, stream=None):
    """SPOT verification with the target's position selection (see sv.h):
    state_logits [B, 1+N, L, V]; parent/node_pos/node_tok [B, N] int32;
    root_mask [B] int64 (bit s: position s is masked in the root state)."""
    B, S, L, V = state_logits.shape
    N = S - 1
    dev = state_logits.device
    code, rs = _rows(state_logits, "state_logits")
    h = handle or default_handle(dev)
    par = _i32(parent, (B, N), "parent", dev) if N > 0 else None
    pos = _i32(node_pos, (B, N), "node_pos", dev) if N > 0 else None
    tok = _i32(node_tok, (B, N), "node_tok", dev) if N > 0 else None
    if (root_mask.dtype != torch.int64 or not root_mask.is_cuda or root_mask.device != dev
            or not root_mask.is_contiguous() or tuple(root_mask.shape) != (B,)):
        raise ValueError("root_mask must be a contiguous int64 CUDA tensor of shape [B]")
    if pos_base is not None and (pos_base.dtype != torch.int64 or not pos_base.is_cuda):
        raise ValueError("pos_base must be an int64 CUDA tensor")
    md = max(N, 1) if max_depth is None else int(max_depth)
    i = lambda *shape: torch.empty(shape, dtype=torch.int32, device=dev)
    out = {"path_len": i(B), "path_nodes": i(B, md), "commit_count": i(B), "commit_pos": i(B),
           "commit_tok": i(B), "match": torch.empty((B, N), dtype=torch.uint8, device=dev),
           "state_pos": i(B, S), "state_tok": i(B, S), "flags": i(B)}
    _check(lib().sv_verify_spot(
        h.ptr, _p(state_logits), code, rs, B, N, L, V, _p(par), _p(pos), _p(tok),
        _p(root_mask), float(T), int(seed) & (2**64 - 1), _p(pos_base), _p(out["path_len"]),
        _p(out["path_nodes"]), md, _p(out["commit_count"]), _p(out["commit_pos"]),
        _p(out["commit_tok"]), _p(out["match"]) if N > 0 else None, _p(out["state_pos"]),
        _p(out["state_tok"]), _p(out["flags"]), _stream(stream, dev)), "sv_verify_spot")
    return out


def sv_packed_anyorder_step(logits, Kv, W, u, win_pos, order, draft, end_pos, *, eos_id=-1,
                            handle=None, stream=None):
    """One any-order Packed-SS iteration (see sv.h); logits [B, Kv + W, V];
    u, end_pos [B]; win_pos, order, draft [B, W] (int32 CUDA tensors)."""
    B, R, V = logits.shape
    if R != Kv + W:
        raise ValueError("logits must be [B, Kv + W, V]")
    dev = logits.device
    code, rs = _rows(logits, "logits")
    h = handle or default_handle(dev)
    uu, end = _i32(u, (B,), "u", dev), _i32(end_pos, (B,), "end_pos", dev)
    wp, od, dr = (_i32(a, (B, W), n, dev) for a, n in ((win_pos, "win_pos"), (order, "order"),
                                                        (draft, "draft")))
    i = lambda *shape: torch.empty(shape, dtype=torch.int32, device=dev)
    out = {"accept_len": i(B), "commit_len": i(B), "commit_pos": i(B, W), "commit_tok": i(B, W),
           "end_pos": i(B), "next_draft": i(B, W),
           "score": torch.empty((B, W), dtype=torch.float32, device=dev)}
    _check(lib().sv_packed_anyorder_step(
        h.ptr, _p(logits), code, rs, B, Kv, W, V, _p(uu), _p(wp), _p(od), _p(dr), _p(end),
        int(eos_id), _p(out["accept_len"]), _p(out["commit_len"]), _p(out["commit_pos"]),
        _p(out["commit_tok"]), _p(out["end_pos"]), _p(out["next_draft"]), _p(out["score"]),
        _stream(stream, dev)), "sv_packed_anyorder_step")
    return out


def sv_packed_step(logits, K, W, prev_draft, prev_len, *, prev_q_at_draft=None,
                   prev_draft_logits=None, prev_q_offset=None, T=0.0, seed=0, it=0,
                   pos_base=None, eos_id=-1, remaining=None, handle=None, stream=None):
    """One Packed-SS iteration; logits [B, K+W, V]."""
    B, R, V = logits.shape
    if R != K + W:
        raise ValueError("logits must be [B, K+W, V]")
    dev = logits.device
    code, rs = _rows(logits, "logits")
    if T > 0:
        code2, rs2 = _rows(prev_draft_logits, "prev_draft_logits")
        if code2 != code or rs2 != rs:
            raise ValueError("prev_draft_logits must match the logits' dtype and row stride")
    h = handle or default_handle(dev)
    pd = _i32(prev_draft, (B, K - 1), "prev_draft", dev) if K > 1 else None
    pl = _i32(prev_len, (B,), "prev_len", dev)
    off = _i32(prev_q_offset, (B,), "prev_q_offset", dev)
    rem = _i32(remaining, (B,), "remaining", dev)
    pq = prev_q_at_draft
    if pq is not None and (pq.dtype != torch.float32 or not pq.is_contiguous()):
        raise ValueError("prev_q_at_draft must be a contiguous float32 tensor")
    out = {"accept_len": torch.empty(B, dtype=torch.int32, device=dev),
           "commit_len": torch.empty(B, dtype=torch.int32, device=dev),
           "committed": torch.empty((B, K), dtype=torch.int32, device=dev),
           "next_draft": torch.empty((B, W), dtype=torch.int32, device=dev),
           "next_len": torch.empty(B, dtype=torch.int32, device=dev),
           "next_q_at_draft": torch.empty((B, W), dtype=torch.float32, device=dev),
           "confidence": torch.empty((B, W), dtype=torch.float32, device=dev),
           "flags": torch.empty(B, dtype=torch.int32, device=dev)}
    _check(lib().sv_packed_step(
        h.ptr, _p(logits), code, rs, B, K, W, V, _p(pd), _p(pl), _p(pq),
        _p(prev_draft_logits) if T > 0 else None, _p(off), float(T), int(seed) & (2**64 - 1),
        int(it) & (2**64 - 1), _p(pos_base), int(eos_id), _p(rem), _p(out["accept_len"]),
        _p(out["commit_len"]), _p(out["committed"]), _p(out["next_draft"]),
        _p(out["next_len"]), _p(out["next_q_at_draft"]), _p(out["confidence"]),
        _p(out["flags"]), _stream(stream, dev)), "sv_packed_step")
    return out


def sv_packed_topk_step(logits, K, W, kp, kq, prev_draft, prev_len, prev_q_ids, prev_q_probs,
                        prev_q_offset, *, T=1.0, seed=0, it=0, pos_base=None, eos_id=-1,
                        remaining=None, handle=None, stream=None):
    """One Packed-SS iteration with top-k truncated target (kp) and drafter
    (kq) distributions; logits [B, K+W, V]; the previous call's drafter lists
    prev_q_ids / prev_q_probs [B, W, kq] (int32 / float32)."""
    B, R, V = logits.shape
    if R != K + W:
        raise ValueError("logits must be [B, K+W, V]")
    dev = logits.device
    code, rs = _rows(logits, "logits")
    h = handle or default_handle(dev)
    pd = _i32(prev_draft, (B, K - 1), "prev_draft", dev) if K > 1 else None
    pl = _i32(prev_len, (B,), "prev_len", dev)
    qi = _i32(prev_q_ids, (B, W, kq), "prev_q_ids", dev)
    off = _i32(prev_q_offset, (B,), "prev_q_offset", dev)
    rem = _i32(remaining, (B,), "remaining", dev)
    qp = prev_q_probs
    if (qp is None or qp.dtype != torch.float32 or not qp.is_contiguous() or
            tuple(qp.shape) != (B, W, kq) or qp.device != dev):
        raise ValueError("prev_q_probs must be a contiguous float32 [B, W, kq] tensor on the "
                         "logits' device")
    out = {"accept_len": torch.empty(B, dtype=torch.int32, device=dev),
           "commit_len": torch.empty(B, dtype=torch.int32, device=dev),
           "committed": torch.empty((B, K), dtype=torch.int32, device=dev),
           "next_draft": torch.empty((B, W), dtype=torch.int32, device=dev),
           "next_len": torch.empty(B, dtype=torch.int32, device=dev),
           "next_q_at_draft": torch.empty((B, W), dtype=torch.float32, device=dev),
           "q_ids": torch.empty((B, W, kq), dtype=torch.int32, device=dev),
           "q_probs": torch.empty((B, W, kq), dtype=torch.float32, device=dev),
           "flags": torch.empty(B, dtype=torch.int32, device=dev)}
    _check(lib().sv_packed_topk_step(
        h.ptr, _p(logits), code, rs, B, K, W, V, int(kp), int(kq), _p(pd), _p(pl), _p(qi),
        _p(qp), _p(off), float(T), int(seed) & (2**64 - 1), int(it) & (2**64 - 1),
        _p(pos_base), int(eos_id), _p(rem), _p(out["accept_len"]), _p(out["commit_len"]),
        _p(out["committed"]), _p(out["next_draft"]), _p(out["next_len"]),
        _p(out["next_q_at_draft"]), _p(out["q_ids"]), _p(out["q_probs"]), _p(out["flags"]),
        _stream(stream, dev)), "sv_packed_topk_step")
    return out

