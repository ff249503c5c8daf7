"""CPU oracle for the tree speculative decoding hot path.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the product library
never does.  It wraps ``jt_oracle.c`` (plain C, fp64 loops) through ctypes and
shares no code with the CUDA path.

Functions return numpy arrays.  See ``jt_oracle.c`` for the definition each
one follows and the passage of the pages it cites.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jt_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_jt_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile jt_oracle.c into a shared library next to it (gcc, -O2)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.jto_topw_lse.argtypes = [P, i64, i64, i32, P, P, P]
            lib.jto_tree_expand.argtypes = [P, P, P, P, i32, i32, i32, P, P, P, P, P, P]
            lib.jto_tree_build.argtypes = [P, P, P, i32, i32, i32, i64, P, P, P, P, P, P, P, P, P]
            lib.jto_tree_attn.argtypes = [P, P, P, i32, P, i32, P, P, P, i32, i32, i32, i32, i32,
                                          dbl, P, i64, P, P]
            lib.jto_verify_accept.argtypes = [P, P, P, P, i32, i32, i64, i32, dbl, P, P, P]
            lib.jto_verify_accept_stochastic.argtypes = [P, P, P, P, P, i32, i32, i64, P, P, P, P,
                                                         P, P, P, P]
            lib.jto_tree_build_mixed.argtypes = [P, P, P, i32, i32, i32, i64, dbl, P, P, P, P, P, P, P]
            lib.jto_tree_expand_capped.argtypes = [P, P, P, P, P, P, i32, i32, i32, P, P, P, P, P, P]
            lib.jto_tree_policy.argtypes = [P, i32, i32, i32, P, i32, i32, i32, i32, i32, i32, dbl, dbl,
                                            dbl, P, P, P, P, P]
            for f in (lib.jto_topw_lse, lib.jto_tree_expand, lib.jto_tree_build,
                      lib.jto_tree_attn, lib.jto_verify_accept, lib.jto_verify_accept_stochastic,
                      lib.jto_tree_build_mixed, lib.jto_tree_expand_capped, lib.jto_tree_policy):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what}: invalid arguments (status {rc})")


def topw_lse(z, W):
    """Per row of z [..., V] fp32: top-W ids, their log-probs and lse (fp64)."""
    z = _c(z, np.float32)
    V = z.shape[-1]
    rows = int(np.prod(z.shape[:-1]))
    tok = np.empty(z.shape[:-1] + (W,), np.int32)
    lp = np.empty(z.shape[:-1] + (W,), np.float64)
    lse = np.empty(z.shape[:-1], np.float64)
    _check(_load().jto_topw_lse(_ptr(z), rows, V, W, _ptr(tok), _ptr(lp), _ptr(lse)), "topw_lse")
    return tok, lp, lse


def _tree_outputs(total):
    return (np.empty(total, np.int32), np.empty(total, np.int32), np.empty(total, np.int32),
            np.empty((total, 8), np.uint32), np.empty(total, np.float64))


def tree_expand(tok, lp, root_token, tree_off, N, W):
    """Best-first expansion from per-depth tables tok/lp [nseq, N, W].

    Returns dict(parent, token, depth, anc, score, gap)."""
    tok, lp = _c(tok, np.int32), _c(lp, np.float64)
    root_token, tree_off = _c(root_token, np.int32), _c(tree_off, np.int32)
    nseq = len(root_token)
    total = int(tree_off[-1])
    parent, token, depth, anc, score = _tree_outputs(total)
    gap = np.empty(nseq, np.float64)
    _check(_load().jto_tree_expand(_ptr(tok), _ptr(lp), _ptr(root_token), _ptr(tree_off), nseq,
                                   N, W, _ptr(parent), _ptr(token), _ptr(depth), _ptr(anc),
                                   _ptr(score), _ptr(gap)), "tree_expand")
    return dict(parent=parent, token=token, depth=depth, anc=anc, score=score, gap=gap)


def tree_expand_capped(tok, lp, root_token, tree_off, N, W, w_cap=None, n_cap=None):
    """tree_expand with optional per-sequence caps: w_cap[b] candidates per
    row, no children below depth n_cap[b]."""
    tok, lp = _c(tok, np.int32), _c(lp, np.float64)
    root_token, tree_off = _c(root_token, np.int32), _c(tree_off, np.int32)
    wc = None if w_cap is None else _c(w_cap, np.int32)
    nc = None if n_cap is None else _c(n_cap, np.int32)
    nseq = len(root_token)
    total = int(tree_off[-1])
    parent, token, depth, anc, score = _tree_outputs(total)
    gap = np.empty(nseq, np.float64)
    _check(_load().jto_tree_expand_capped(_ptr(tok), _ptr(lp), _ptr(root_token), _ptr(tree_off),
                                          _ptr(wc), _ptr(nc), nseq, N, W, _ptr(parent), _ptr(token),
                                          _ptr(depth), _ptr(anc), _ptr(score), _ptr(gap)),
           "tree_expand_capped")
    return dict(parent=parent, token=token, depth=depth, anc=anc, score=score, gap=gap)


POLICY_DEFAULTS = dict(b_min=16, b_max=256, node_cap=0, w_min=2, n_min=2, n_slack=3, beta=0.25,
                       log_conf=float(np.log(0.5)), acc_thresh=3.0)


def tree_policy(lp, accept_len, budget_state, acc_ema, **params):
    """One step of the adaptive tree policy (see jt_oracle.c).  lp is the
    per-depth table [nseq, N, W]; accept_len [nseq] (-1 = not observed) or
    None.  Returns dict(tree_off, w_cap, n_cap, budget_state, acc_ema) with
    the updated state (the inputs are not modified)."""
    p = dict(POLICY_DEFAULTS)
    p.update(params)
    lp = _c(lp, np.float64)
    nseq, N, W = lp.shape
    acc = None if accept_len is None else _c(accept_len, np.int32)
    bs = np.array(budget_state, dtype=np.int32, copy=True)
    ema = np.array(acc_ema, dtype=np.float64, copy=True)
    off = np.empty(nseq + 1, np.int32)
    wc = np.empty(nseq, np.int32)
    nc = np.empty(nseq, np.int32)
    _check(_load().jto_tree_policy(_ptr(lp), nseq, N, W, _ptr(acc), p["b_min"], p["b_max"], p["node_cap"],
                                   p["w_min"], p["n_min"], p["n_slack"], float(p["beta"]),
                                   float(p["log_conf"]), float(p["acc_thresh"]), _ptr(bs), _ptr(ema),
                                   _ptr(off), _ptr(wc), _ptr(nc)), "tree_policy")
    return dict(tree_off=off, w_cap=wc, n_cap=nc, budget_state=bs, acc_ema=ema)


def tree_build(draft_logits, root_token, tree_off, W):
    """Full tree build from per-depth draft logits [nseq, N, V] fp32.

    Returns dict(parent, token, depth, anc, score, gap, tok, lp, lse)."""
    z = _c(draft_logits, np.float32)
    nseq, N, V = z.shape
    root_token, tree_off = _c(root_token, np.int32), _c(tree_off, np.int32)
    total = int(tree_off[-1])
    parent, token, depth, anc, score = _tree_outputs(total)
    gap = np.empty(nseq, np.float64)
    tok = np.empty((nseq, N, W), np.int32)
    lp = np.empty((nseq, N, W), np.float64)
    lse = np.empty((nseq, N), np.float64)
    _check(_load().jto_tree_build(_ptr(z), _ptr(root_token), _ptr(tree_off), nseq, N, W, V,
                                  _ptr(parent), _ptr(token), _ptr(depth), _ptr(anc), _ptr(score),
                                  _ptr(gap), _ptr(tok), _ptr(lp), _ptr(lse)), "tree_build")
    return dict(parent=parent, token=token, depth=depth, anc=anc, score=score, gap=gap,
                tok=tok, lp=lp, lse=lse)


def tree_build_mixed(draft_logits, root_token, tree_off, W, alpha):
    """Tree build whose step from depth d to d+1 scores
    (1 - alpha) * log-prob - alpha * entropy(draft row d), alpha in [0, 1]
    (1: pure entropy score); a candidate of probability 0 stays at -inf.

    Returns dict(parent, token, depth, anc, score, gap, entropy [nseq, N])."""
    z = _c(draft_logits, np.float32)
    nseq, N, V = z.shape
    root_token, tree_off = _c(root_token, np.int32), _c(tree_off, np.int32)
    total = int(tree_off[-1])
    parent, token, depth, anc, score = _tree_outputs(total)
    gap = np.empty(nseq, np.float64)
    ent = np.empty((nseq, N), np.float64)
    _check(_load().jto_tree_build_mixed(_ptr(z), _ptr(root_token), _ptr(tree_off), nseq, N, W, V,
                                        float(alpha), _ptr(parent), _ptr(token), _ptr(depth), _ptr(anc),
                                        _ptr(score), _ptr(gap), _ptr(ent)), "tree_build_mixed")
    return dict(parent=parent, token=token, depth=depth, anc=anc, score=score, gap=gap, entropy=ent)


def tree_attn(q, k_cache, v_cache, block_table, prefix_len, tree_off, parent, scale, rows=None):
    """Tree-causal paged attention in fp64.

    q [total, Hq, D], k/v [pages, page_size, Hkv, D] given as numpy float32
    arrays (dtype 0) or uint16 bf16 bit patterns (dtype 1).  Returns
    (out [n, Hq, D] float64, lse [n, Hq] float64) for the nodes in ``rows``
    (global indices; default all)."""
    if q.dtype == np.uint16:
        dtype = 1
    elif q.dtype == np.float32:
        dtype = 0
    else:
        raise TypeError("q/k/v must be float32 or uint16 (bf16 bits)")
    q, k_cache, v_cache = (np.ascontiguousarray(a) for a in (q, k_cache, v_cache))
    assert k_cache.dtype == q.dtype and v_cache.dtype == q.dtype
    block_table = _c(block_table, np.int32)
    prefix_len, tree_off, parent = (_c(a, np.int32) for a in (prefix_len, tree_off, parent))
    total, Hq, D = q.shape
    _, page_size, Hkv, _ = k_cache.shape
    nseq, max_pages = block_table.shape
    if rows is None:
        n = total
        rows_p = None
    else:
        rows = _c(rows, np.int32)
        n = len(rows)
        rows_p = _ptr(rows)
    out = np.empty((n, Hq, D), np.float64)
    lse = np.empty((n, Hq), np.float64)
    _check(_load().jto_tree_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), dtype, _ptr(block_table),
                                 max_pages, _ptr(prefix_len), _ptr(tree_off), _ptr(parent), nseq,
                                 Hq, Hkv, D, page_size, float(scale), rows_p, n, _ptr(out),
                                 _ptr(lse)), "tree_attn")
    return out, lse


def verify_accept(target_logits, parent, token, tree_off, N, rule, log_t=0.0):
    """Tree acceptance; rule 0 = greedy, 1 = margin (log_t = log(t)).

    Returns (accept_len [nseq], path [nseq, N+1], bonus [nseq])."""
    z = _c(target_logits, np.float32)
    V = z.shape[-1]
    parent, token, tree_off = (_c(a, np.int32) for a in (parent, token, tree_off))
    nseq = len(tree_off) - 1
    acc = np.empty(nseq, np.int32)
    path = np.empty((nseq, N + 1), np.int32)
    bonus = np.empty(nseq, np.int32)
    _check(_load().jto_verify_accept(_ptr(z), _ptr(parent), _ptr(token), _ptr(tree_off), nseq, N,
                                     V, rule, float(log_t), _ptr(acc), _ptr(path), _ptr(bonus)),
           "verify_accept")
    return acc, path, bonus

def verify_accept_stochastic(target_logits, draft_logits, parent, token, tree_off, N, u_accept,
                             u_bonus, with_residual=False):
    """Temperature-1 speculative-sampling acceptance over the tree with the
    caller's uniforms.  Returns (accept_len, path, bonus, min_margin), and
    with with_residual=True also (final_r [nseq, V], final_u [nseq]): the
    normalised residual each bonus was drawn from and the draw's uniform."""
    z = _c(target_logits, np.float32)
    V = z.shape[-1]
    dz = _c(draft_logits, np.float32) if draft_logits is not None else None
    parent, token, tree_off = (_c(a, np.int32) for a in (parent, token, tree_off))
    ua, ub = _c(u_accept, np.float64), _c(u_bonus, np.float64)
    nseq = len(tree_off) - 1
    acc = np.empty(nseq, np.int32)
    path = np.empty((nseq, N + 1), np.int32)
    bonus = np.empty(nseq, np.int32)
    margin = np.empty(nseq, np.float64)
    fr = np.empty((nseq, V), np.float64) if with_residual else None
    fu = np.empty(nseq, np.float64) if with_residual else None
    _check(_load().jto_verify_accept_stochastic(_ptr(z), _ptr(dz) if dz is not None else None,
                                                _ptr(parent), _ptr(token), _ptr(tree_off), nseq, N,
                                                V, _ptr(ua), _ptr(ub), _ptr(acc), _ptr(path),
                                                _ptr(bonus), _ptr(margin), _ptr(fr), _ptr(fu)),
           "verify_accept_stochastic")
    if with_residual:
        return acc, path, bonus, margin, fr, fu
    return acc, path, bonus, margin
