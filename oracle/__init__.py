"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle for draft-block verification.

A plain, slow restatement of what the CUDA library computes, written from the
three source pages (see the header of ``sv_oracle.c`` for the citations and
the readings).  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  It shares no code with
``draft_block_verification_gb300``; the only module both sides use is
``datagen`` (seeded inputs, none of the method's arithmetic).

Logit arrays are numpy arrays: ``float32`` for fp32 rows, ``uint16`` holding
the raw bit patterns for bf16 rows.  Every function returns numpy arrays;
probabilities, log-sum-exps and total variations are fp64.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIBPATH = os.path.join(_LIBDIR, "liboracle.so")
_lib = None

LOSSLESS, RATIO, LINEAR, CACTUS = 0, 1, 2, 3
ST_ACCEPT, ST_SAMPLE, ST_DRAFT, ST_TREE = 1, 2, 3, 4
FLAG_EPS = 1e-9


def build(force: bool = False) -> str:
    """Compile sv_oracle.c with gcc (fp64, no fast-math) into oracle/_lib."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIBPATH)
            and os.path.getmtime(_LIBPATH) >= os.path.getmtime(_SRC)):
        return _LIBPATH
    tmp = _LIBPATH + ".%d.tmp" % os.getpid()
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", "-o", tmp, _SRC]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIBPATH)
    return _LIBPATH


def _L():
    global _lib
    if _lib is None:
        lib = C.CDLL(build())
        u64, u32, i64, i32, dbl = C.c_uint64, C.c_uint32, C.c_int64, C.c_int, C.c_double
        vp = C.c_void_p
        lib.or_mix64.restype, lib.or_mix64.argtypes = u64, [u64]
        lib.or_key.restype, lib.or_key.argtypes = u64, [u64, u32, u64, i64, u64]
        lib.or_fine52.restype, lib.or_fine52.argtypes = u64, [u64, u32]
        lib.or_is_top.restype, lib.or_is_top.argtypes = i32, [u64, u32]
        lib.or_skip_threshold.restype, lib.or_skip_threshold.argtypes = u64, [i32]
        lib.or_row_uniforms.restype, lib.or_row_uniforms.argtypes = None, [u64, i32, vp, vp]
        lib.or_uniform.restype, lib.or_uniform.argtypes = dbl, [u64, u32]
        lib.or_gumbel.restype, lib.or_gumbel.argtypes = dbl, [u64, u32]
        lib.or_lse.restype, lib.or_lse.argtypes = dbl, [vp, i32, dbl]
        lib.or_argmax.restype, lib.or_argmax.argtypes = i32, [vp, i32]
        lib.or_gumbel_argmax.restype = i32
        lib.or_gumbel_argmax.argtypes = [vp, i32, u64, vp]
        lib.or_accept_prob.restype = dbl
        lib.or_accept_prob.argtypes = [dbl, dbl, i32, dbl]
        lib.or_residual_weights.restype = None
        lib.or_residual_weights.argtypes = [vp, vp, i32, dbl, dbl, dbl, dbl, i32, dbl, dbl, vp]
        lib.or_cactus_gamma.restype, lib.or_cactus_gamma.argtypes = dbl, [dbl, dbl]
        lib.or_residual_scale.restype = dbl
        lib.or_residual_scale.argtypes = [dbl, i32, dbl]
        lib.or_tv.restype, lib.or_tv.argtypes = dbl, [vp, vp, i32, dbl, dbl, dbl, dbl]
        lib.or_verify_greedy.restype = i32
        lib.or_verify_greedy.argtypes = [vp, i32, i64, i32, i32, i32, vp, vp, vp, vp]
        lib.or_verify_sample.restype = i32
        lib.or_verify_sample.argtypes = [vp, vp, i32, i64, i32, i32, i32, vp, vp, dbl, dbl,
                                         i32, dbl, u64, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.or_verify_tree.restype = i32
        lib.or_verify_tree.argtypes = [vp, i32, i64, i32, i32, i32, vp, vp, vp, dbl, u64, vp,
                                       vp, vp, i32, vp, vp, vp]
        lib.or_packed_step.restype = i32
        lib.or_packed_step.argtypes = [vp, i32, i64, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                       dbl, u64, u64, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                       vp]
        lib.or_verify_spot.restype = i32
        lib.or_verify_spot.argtypes = [vp, i32, i64, i32, i32, i32, i32, vp, vp, vp, vp, dbl,
                                       u64, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.or_packed_anyorder_step.restype = i32
        lib.or_packed_anyorder_step.argtypes = [vp, i32, i64, i32, i32, i32, i32, vp, vp, vp, vp,
                                                vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.or_packed_topk_step.restype = i32
        lib.or_packed_topk_step.argtypes = [vp, i32, i64, i32, i32, i32, i32, i32, i32, vp, vp,
                                            vp, vp, vp, dbl, u64, u64, vp, i32, vp, vp, vp, vp,
                                            vp, vp, vp, vp, vp, vp]
        lib.or_topk.restype = None
        lib.or_topk.argtypes = [vp, i32, i32, vp]
        lib.or_num_threads.restype, lib.or_num_threads.argtypes = i32, []
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def f32(x: float) -> float:
    """The value a C ``float`` parameter carries (temperatures and lambda are
    passed to the library as fp32; the oracle uses the same numbers)."""
    return float(np.float32(x))


def _dtype_code(logits: np.ndarray) -> int:
    if logits.dtype == np.float32:
        return 0
    if logits.dtype == np.uint16:
        return 1
    raise TypeError("logits must be float32 or uint16 (bf16 bit patterns)")


def _i32(a, shape=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.int32)
    if shape is not None:
        a = a.reshape(shape)
    return a


def _i64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int64)


def num_threads() -> int:
    return int(_L().or_num_threads())


# --- counter RNG -------------------------------------------------------------

def mix64(x: int) -> int:
    return int(_L().or_mix64(x & (2**64 - 1)))


def key(seed: int, stream: int, seq: int, pos: int, it: int = 0) -> int:
    return int(_L().or_key(seed & (2**64 - 1), stream, seq & (2**64 - 1), pos, it & (2**64 - 1)))


def fine52(k: int, v: int) -> int:
    """The 52 fine bits m of id v: w = (2m + 1) / 2^53."""
    return int(_L().or_fine52(k, v))


def is_top(k: int, v: int) -> bool:
    """Whether id v falls in the top 1/256 of the unit interval under key k."""
    return bool(_L().or_is_top(k, v))


def skip_threshold(g: int) -> int:
    """C_g = ceil(2^64 (255/256)^g), the skip thresholds (g = 1..256)."""
    return int(_L().or_skip_threshold(g))


def uniform(k: int, v: int) -> float:
    return float(_L().or_uniform(k, v))


def row_uniforms(k: int, V: int):
    """(u[V], top[V]) of ids 0..V-1 under key k."""
    u = np.empty(V)
    top = np.empty(V, np.uint8)
    _L().or_row_uniforms(k, V, _p(u), _p(top))
    return u, top.astype(bool)


def gumbel(k: int, v: int) -> float:
    return float(_L().or_gumbel(k, v))


# --- row primitives ------------------------------------------------------------

def lse(x, T: float) -> float:
    x = np.ascontiguousarray(x, dtype=np.float64)
    return float(_L().or_lse(_p(x), x.size, float(T)))


def argmax(x) -> int:
    x = np.ascontiguousarray(x, dtype=np.float64)
    return int(_L().or_argmax(_p(x), x.size))


def gumbel_argmax(score, k: int):
    """(index, gap) of argmax_v score[v] + G(k, v); -inf entries are skipped."""
    s = np.ascontiguousarray(score, dtype=np.float64)
    gap = np.zeros(1, dtype=np.float64)
    idx = int(_L().or_gumbel_argmax(_p(s), s.size, k, _p(gap)))
    return idx, float(gap[0])


def accept_prob(log_p: float, log_q: float, mode: int = LOSSLESS, lam: float = 1.0) -> float:
    return float(_L().or_accept_prob(log_p, log_q, mode, lam))


def cactus_gamma(p: float, delta: float) -> float:
    """gamma*: the modified Cactus target probability of the drafted token."""
    return float(_L().or_cactus_gamma(float(p), float(delta)))


def residual_scale(log_pd: float, mode: int = LOSSLESS, lam: float = 1.0) -> float:
    """c = (1 - gamma*) / (1 - p(d)) for CACTUS (1 for the other modes)."""
    return float(_L().or_residual_scale(float(log_pd), int(mode), float(lam)))


def residual_weights(x, y, Tp: float, Tq: float, mode: int = LOSSLESS, lam: float = 1.0,
                     d: int = None):
    """Unnormalised residual weights for target logits x and drafter logits y
    (d: the rejected draft token, which the CACTUS weights depend on)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.ascontiguousarray(y, dtype=np.float64)
    w = np.empty_like(x)
    Lp, Lq = lse(x, Tp), lse(y, Tq)
    c = 1.0 if d is None else residual_scale(x[d] / Tp - Lp, mode, lam)
    _L().or_residual_weights(_p(x), _p(y), x.size, Tp, Tq, Lp, Lq, mode, lam, c, _p(w))
    return w


def tv(x, y, Tp: float, Tq: float) -> float:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.ascontiguousarray(y, dtype=np.float64)
    return float(_L().or_tv(_p(x), _p(y), x.size, Tp, Tq, lse(x, Tp), lse(y, Tq)))


# --- the four verify procedures ------------------------------------------------

def verify_greedy(target, draft_ids, draft_len=None):
    """target [B, K+1, V]; draft_ids [B, K]; draft_len [B] or None (= K)."""
    target = np.ascontiguousarray(target)
    B, K1, V = target.shape
    K = K1 - 1
    ids = _i32(draft_ids, (B, K))
    dl = _i32(draft_len)
    acc = np.empty(B, np.int32)
    nxt = np.empty(B, np.int32)
    rc = _L().or_verify_greedy(_p(target), _dtype_code(target), V, B, K, V, _p(ids), _p(dl),
                               _p(acc), _p(nxt))
    if rc:
        raise ValueError("oracle: invalid greedy inputs")
    return {"accept_len": acc, "next_token": nxt}


def verify_sample(target, draft, draft_ids, draft_len=None, T_p=1.0, T_q=1.0, mode=LOSSLESS,
                  lam=1.0, seed=0, pos_base=None, want_tv=True):
    """target [B, K+1, V], draft [B, K, V] (same dtype); see sv_oracle.c."""
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    B, K1, V = target.shape
    K = K1 - 1
    if draft.dtype != target.dtype or draft.shape != (B, K, V):
        raise ValueError("draft must be [B, K, V] with the target's dtype")
    ids = _i32(draft_ids, (B, K))
    dl = _i32(draft_len)
    pb = _i64(pos_base)
    out = {
        "accept_len": np.empty(B, np.int32), "next_token": np.empty(B, np.int32),
        "p_at_draft": np.empty((B, K)), "q_at_draft": np.empty((B, K)),
        "lse_p": np.empty((B, K + 1)), "lse_q": np.empty((B, K)),
        "tv": np.empty((B, K)) if want_tv else None, "flags": np.empty(B, np.int32),
    }
    rc = _L().or_verify_sample(
        _p(target), _p(draft), _dtype_code(target), V, B, K, V, _p(ids), _p(dl), f32(T_p),
        f32(T_q), int(mode), f32(lam), int(seed) & (2**64 - 1), _p(pb),
        _p(out["accept_len"]), _p(out["next_token"]), _p(out["p_at_draft"]),
        _p(out["q_at_draft"]), _p(out["lse_p"]), _p(out["lse_q"]), _p(out["tv"]),
        _p(out["flags"]))
    if rc:
        raise ValueError("oracle: invalid sample inputs")
    if not want_tv:
        del out["tv"]
    return out


def verify_tree(node_logits, parent, node_pos, node_tok, T=0.0, seed=0, pos_base=None,
                max_depth=None):
    """node_logits [B, N, V]; parent/node_pos/node_tok [B, N]."""
    node_logits = np.ascontiguousarray(node_logits)
    B, N, V = node_logits.shape
    par, pos, tok = _i32(parent, (B, N)), _i32(node_pos, (B, N)), _i32(node_tok, (B, N))
    if max_depth is None:
        max_depth = max(N, 1)
    pb = _i64(pos_base)
    out = {
        "path_len": np.empty(B, np.int32), "path_nodes": np.empty((B, max_depth), np.int32),
        "commit_count": np.empty(B, np.int32), "match": np.empty((B, N), np.uint8),
        "flags": np.empty(B, np.int32),
    }
    rc = _L().or_verify_tree(
        _p(node_logits), _dtype_code(node_logits), V, B, N, V, _p(par), _p(pos), _p(tok),
        f32(T), int(seed) & (2**64 - 1), _p(pb), _p(out["path_len"]), _p(out["path_nodes"]),
        int(max_depth), _p(out["commit_count"]), _p(out["match"]), _p(out["flags"]))
    if rc:
        raise ValueError("oracle: invalid tree inputs")
    return out


def packed_step(logits, K, W, prev_draft, prev_len, prev_q_at_draft=None,
                prev_draft_logits=None, prev_q_offset=None, T=0.0, seed=0, it=0,
                pos_base=None, eos_id=-1, remaining=None):
    """logits [B, K+W, V]; prev_draft [B, K-1]; see sv_oracle.c."""
    logits = np.ascontiguousarray(logits)
    B, R, V = logits.shape
    if R != K + W or K < 1:
        raise ValueError("logits must be [B, K+W, V] with K >= 1")
    pd = _i32(prev_draft, (B, K - 1))
    pl = _i32(prev_len)
    pq = None if prev_q_at_draft is None else np.ascontiguousarray(prev_q_at_draft,
                                                                   dtype=np.float32)
    pdl = None if prev_draft_logits is None else np.ascontiguousarray(prev_draft_logits)
    if T > 0 and (pq is None or pdl is None or pdl.dtype != logits.dtype):
        raise ValueError("T > 0 needs prev_q_at_draft and prev_draft_logits")
    off = _i32(prev_q_offset)
    pb = _i64(pos_base)
    rem = _i32(remaining)
    out = {
        "accept_len": np.empty(B, np.int32), "commit_len": np.empty(B, np.int32),
        "committed": np.empty((B, K), np.int32), "next_draft": np.empty((B, W), np.int32),
        "next_len": np.empty(B, np.int32), "next_q_at_draft": np.empty((B, W)),
        "confidence": np.empty((B, W)), "flags": np.empty(B, np.int32),
    }
    rc = _L().or_packed_step(
        _p(logits), _dtype_code(logits), V, B, K, W, V, _p(pd), _p(pl), _p(pq), _p(pdl),
        _p(off), f32(T), int(seed) & (2**64 - 1), int(it) & (2**64 - 1), _p(pb), int(eos_id),
        _p(rem), _p(out["accept_len"]), _p(out["commit_len"]), _p(out["committed"]),
        _p(out["next_draft"]), _p(out["next_len"]), _p(out["next_q_at_draft"]),
        _p(out["confidence"]), _p(out["flags"]))
    if rc:
        raise ValueError("oracle: invalid packed-step inputs")
    return out


def topk(x, k):
    """The k largest entries of the fp64 row x (ties to the lowest id), in
    that order."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    ids = np.empty(k, np.int32)
    _L().or_topk(_p(x), x.shape[0], int(k), _p(ids))
    return ids


def packed_topk_step(logits, K, W, kp, kq, prev_draft, prev_len, prev_q_ids, prev_q_probs,
                     prev_q_offset, T, seed=0, it=0, pos_base=None, eos_id=-1, remaining=None):
    """Packed-SS step with top-k truncated target (kp) and drafter (kq)
    distributions; prev_q_ids / prev_q_probs [B, W, kq]; see sv_oracle.c."""
    logits = np.ascontiguousarray(logits)
    B, R, V = logits.shape
    if R != K + W or K < 1:
        raise ValueError("logits must be [B, K+W, V] with K >= 1")
    pd = _i32(prev_draft, (B, K - 1))
    pl = _i32(prev_len)
    qi = _i32(prev_q_ids, (B, W, kq))
    qp = np.ascontiguousarray(prev_q_probs, dtype=np.float32).reshape(B, W, kq)
    off = _i32(prev_q_offset)
    pb = _i64(pos_base)
    rem = _i32(remaining)
    out = {
        "accept_len": np.empty(B, np.int32), "commit_len": np.empty(B, np.int32),
        "committed": np.empty((B, K), np.int32), "next_draft": np.empty((B, W), np.int32),
        "next_len": np.empty(B, np.int32), "next_q_at_draft": np.empty((B, W)),
        "q_ids": np.empty((B, W, kq), np.int32), "q_probs": np.empty((B, W, kq)),
        "flags": np.empty(B, np.int32),
    }
    rc = _L().or_packed_topk_step(
        _p(logits), _dtype_code(logits), V, B, K, W, V, int(kp), int(kq), _p(pd), _p(pl),
        _p(qi), _p(qp), _p(off), f32(T), int(seed) & (2**64 - 1), int(it) & (2**64 - 1),
        _p(pb), int(eos_id), _p(rem), _p(out["accept_len"]), _p(out["commit_len"]),
        _p(out["committed"]), _p(out["next_draft"]), _p(out["next_len"]),
        _p(out["next_q_at_draft"]), _p(out["q_ids"]), _p(out["q_probs"]), _p(out["flags"]))
    if rc:
        raise ValueError("oracle: invalid truncated packed-step inputs")
    return out


def verify_spot(state_logits, parent, node_pos, node_tok, root_mask, T=0.0, seed=0,
                pos_base=None, max_depth=None):
    """SPOT state-equality verification with the target's position selection.
    state_logits [B, 1+N, L, V]; parent/node_pos/node_tok [B, N]; root_mask [B]
    (bit s set: block position s is masked in the root state)."""
    state_logits = np.ascontiguousarray(state_logits)
    B, S, L, V = state_logits.shape
    N = S - 1
    par, pos, tok = (_i32(a, (B, N)) for a in (parent, node_pos, node_tok))
    rm = np.ascontiguousarray(np.asarray(root_mask, dtype=np.uint64).reshape(B))
    if max_depth is None:
        max_depth = max(N, 1)
    pb = _i64(pos_base)
    out = {
        "path_len": np.empty(B, np.int32), "path_nodes": np.empty((B, max_depth), np.int32),
        "commit_count": np.empty(B, np.int32), "commit_pos": np.empty(B, np.int32),
        "commit_tok": np.empty(B, np.int32), "match": np.empty((B, max(N, 1)), np.uint8),
        "state_pos": np.empty((B, S), np.int32), "state_tok": np.empty((B, S), np.int32),
        "flags": np.empty(B, np.int32),
    }
    rc = _L().or_verify_spot(
        _p(state_logits), _dtype_code(state_logits), V, B, N, L, V, _p(par), _p(pos), _p(tok),
        _p(rm), f32(T), int(seed) & (2**64 - 1), _p(pb), _p(out["path_len"]),
        _p(out["path_nodes"]), int(max_depth), _p(out["commit_count"]), _p(out["commit_pos"]),
        _p(out["commit_tok"]), _p(out["match"]), _p(out["state_pos"]), _p(out["state_tok"]),
        _p(out["flags"]))
    if rc:
        raise ValueError("oracle: invalid SPOT tree inputs")
    out["match"] = out["match"][:, :N]
    return out


def packed_anyorder_step(logits, Kv, W, u, win_pos, order, draft, end_pos, eos_id=-1):
    """One any-order Packed-SS iteration (greedy); logits [B, Kv + W, V];
    u [B]; win_pos, order, draft [B, W]; end_pos [B].  See sv_oracle.c."""
    logits = np.ascontiguousarray(logits)
    B, R, V = logits.shape
    if R != Kv + W:
        raise ValueError("logits must be [B, Kv + W, V]")
    u, end = _i32(u, (B,)), _i32(end_pos, (B,))
    wp, od, dr = (_i32(a, (B, W)) for a in (win_pos, order, draft))
    out = {"accept_len": np.empty(B, np.int32), "commit_len": np.empty(B, np.int32),
           "commit_pos": np.empty((B, W), np.int32), "commit_tok": np.empty((B, W), np.int32),
           "end_pos": np.empty(B, np.int32), "next_draft": np.empty((B, W), np.int32),
           "score": np.empty((B, W)), "next_order": np.empty((B, W), np.int32)}
    rc = _L().or_packed_anyorder_step(
        _p(logits), _dtype_code(logits), V, B, Kv, W, V, _p(u), _p(wp), _p(od), _p(dr), _p(end),
        int(eos_id), _p(out["accept_len"]), _p(out["commit_len"]), _p(out["commit_pos"]),
        _p(out["commit_tok"]), _p(out["end_pos"]), _p(out["next_draft"]), _p(out["score"]),
        _p(out["next_order"]))
    if rc:
        raise ValueError("oracle: invalid any-order step inputs")
    return out
