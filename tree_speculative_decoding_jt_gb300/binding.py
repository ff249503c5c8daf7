"""Thin ctypes binding of libjt (include/jt.h) for torch tensors.

Argument marshalling only: every step runs in the library's CUDA kernels.
Each function takes CUDA tensors, passes their device pointers and the
current torch stream to the C entry point of the same name, and raises
``JtError`` on a non-OK status.  Workspaces and outputs are allocated with
torch when the caller does not pass them.  There is no CPU path: without a
GPU or without the built library the calls fail.
"""
from __future__ import annotations

import ctypes
import functools
import math
import os
import threading

import torch

from . import build as _build

JT_OK, JT_ERR_INVALID, JT_ERR_UNSUPPORTED, JT_ERR_CUDA, JT_ERR_TIMEOUT, JT_ERR_WORKSPACE = 0, -1, -2, -3, -4, -5
JT_DTYPE_F32, JT_DTYPE_BF16 = 0, 1
JT_RULE_GREEDY, JT_RULE_MARGIN = 0, 1
(JT_OP_TREE_BUILD, JT_OP_TREE_ATTN, JT_OP_VERIFY_ACCEPT, JT_OP_TREE_TOPW, JT_OP_TREE_BUILD_MIXED,
 JT_OP_TREE_POLICY) = 0, 1, 2, 3, 4, 5
JT_MAX_TREE, JT_MAX_W, JT_MAX_N, JT_PAGE_SIZE = 256, 8, 64, 16

# every symbol include/jt.h declares
EXPORTS = ("jt_workspace_size", "jt_tree_build", "jt_tree_topw", "jt_tree_expand",
           "jt_tree_attn_paged", "jt_verify_accept", "jt_check", "jt_status_str", "jt_version",
           "jt_tree_build_noalloc", "jt_verify_accept_stochastic", "jt_tree_build_mixed",
           "jt_tree_expand_capped", "jt_tree_policy", "jt_tree_build_adaptive", "jt_selftest_wait_timeout")

_lock = threading.Lock()
_lib = None


class PolicyParams(ctypes.Structure):
    """jt_policy_params of include/jt.h (field order and types as there)."""
    _fields_ = [("b_min", ctypes.c_int32), ("b_max", ctypes.c_int32), ("node_cap", ctypes.c_int32),
                ("w_min", ctypes.c_int32), ("n_min", ctypes.c_int32), ("n_slack", ctypes.c_int32),
                ("beta", ctypes.c_double), ("log_conf", ctypes.c_double), ("acc_thresh", ctypes.c_double)]


def policy_params(b_min=16, b_max=256, node_cap=0, w_min=2, n_min=2, n_slack=3, beta=0.25,
                  log_conf=-0.6931471805599453, acc_thresh=3.0) -> PolicyParams:
    """Policy parameters with the defaults used by the tests and bench.py."""
    return PolicyParams(b_min, b_max, node_cap, w_min, n_min, n_slack, float(beta), float(log_conf),
                        float(acc_thresh))


def policy_ceiling(params: PolicyParams, nseq: int) -> int:
    """Per-request budget ceiling of the policy (min(b_max, max(b_min,
    node_cap // nseq)) with a node cap, else b_max)."""
    if params.node_cap > 0:
        return min(params.b_max, max(params.b_min, params.node_cap // nseq))
    return params.b_max


class JtError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {jt_status_str(status)}")


def library_variant() -> str:
    """The library variant this process loads: JT_LIB_VARIANT ("" = the
    default build, "checks" = extra device-side input checks and NVTX
    ranges)."""
    return os.environ.get("JT_LIB_VARIANT", "")


def library_path() -> str:
    return _build.lib_path(library_variant())


def load(build_if_missing: bool = True):
    """Load libjt (building it with nvcc first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        variant = library_variant()
        path = _build.build(variant=variant) if build_if_missing else _build.lib_path(variant)
        if not os.path.exists(path):
            raise RuntimeError(f"libjt.so not found at {path}; run tree_speculative_decoding_jt_gb300.build")
        lib = ctypes.CDLL(path)
        P, i32, i64, f32, f64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                     ctypes.c_double, ctypes.c_size_t)
        lib.jt_workspace_size.argtypes = [i32, i32, i32, i32, i64, i32, i32, i32, i32, i32, i32]
        lib.jt_workspace_size.restype = sz
        lib.jt_tree_build.argtypes = [P, P, P, i32, i32, i32, i64, i32, P, P, P, P, P, sz, P]
        lib.jt_tree_build_mixed.argtypes = [P, P, P, i32, i32, i32, i64, i32, f64, P, P, P, P, P, sz, P]
        lib.jt_tree_topw.argtypes = [P, i64, i64, i32, P, P, P, P, sz, P]
        lib.jt_tree_build_noalloc.argtypes = [P, P, P, i32, i32, i32, i64, i32, P, P, P, P, i32, P]
        lib.jt_tree_expand.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, P, P, P, sz, P]
        lib.jt_tree_expand_capped.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, P, P, P, P, P, sz, P]
        lib.jt_tree_policy.argtypes = [P, i32, i32, i32, P, ctypes.POINTER(PolicyParams), P, P, P, P, P, P,
                                       sz, P]
        lib.jt_tree_build_adaptive.argtypes = [P, P, i32, i32, i32, i64, i32, P, ctypes.POINTER(PolicyParams),
                                               P, P, P, P, P, P, P, P, P, P, sz, P]
        lib.jt_tree_attn_paged.argtypes = [P, P, P, i32, P, i32, i32, P, P, P, i32, i32, i32, i32,
                                           i32, i32, i32, f32, P, P, P, sz, P]
        lib.jt_verify_accept.argtypes = [P, P, P, P, i32, i32, i64, i32, i32, f64, P, P, P, P, sz, P]
        lib.jt_verify_accept_stochastic.argtypes = [P, P, P, P, P, i32, i32, i64, i32, P, P, P, P, P,
                                                    P, sz, P]
        lib.jt_check.argtypes = [P, P]
        lib.jt_selftest_wait_timeout.argtypes = [P, sz, P]
        lib.jt_status_str.argtypes = [i32]
        lib.jt_status_str.restype = ctypes.c_char_p
        lib.jt_version.argtypes = []
        for name in ("jt_tree_build", "jt_tree_topw", "jt_tree_expand", "jt_tree_attn_paged",
                     "jt_verify_accept", "jt_check", "jt_version", "jt_tree_build_noalloc",
                     "jt_verify_accept_stochastic", "jt_tree_build_mixed", "jt_tree_expand_capped",
                     "jt_tree_policy", "jt_tree_build_adaptive", "jt_selftest_wait_timeout"):
            getattr(lib, name).restype = i32
        _lib = lib
        return lib


def jt_status_str(status: int) -> str:
    return load().jt_status_str(int(status)).decode()


def jt_version() -> int:
    return int(load().jt_version())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libjt has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _check(rc, where):
    if rc != JT_OK:
        raise JtError(rc, where)


def _tensors(obj):
    if isinstance(obj, torch.Tensor):
        yield obj
    elif isinstance(obj, (tuple, list)):
        for o in obj:
            yield from _tensors(o)


def _on_tensor_device(fn):
    """Run a binding call with its tensors' device current.  The library
    launches on the current device (its stream, its per-device set-up and
    fixed scratch), so a call whose tensors live on another device than the
    current one is moved there; tensors on different devices are refused."""
    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        devs = {t.device for t in _tensors(list(args) + list(kwargs.values())) if t.is_cuda}
        if len(devs) > 1:
            raise ValueError(f"{fn.__name__}: tensors on several devices ({sorted(map(str, devs))})")
        if not devs:
            return fn(*args, **kwargs)
        with torch.cuda.device(devs.pop()):
            return fn(*args, **kwargs)
    return wrapper


def jt_workspace_size(op, nseq=0, N=0, W=0, V=0, total_nodes=0, Hq=0, Hkv=0, D=0, max_pages=0,
                      max_tree=0) -> int:
    return int(load().jt_workspace_size(op, nseq, N, W, V, total_nodes, Hq, Hkv, D, max_pages,
                                        max_tree))


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zeroed device buffer usable as a libjt workspace (torch allocations
    are 256-byte aligned; the library needs the header zero before first
    use)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


@_on_tensor_device
def jt_verify_accept_stochastic(target_logits, draft_logits, parent, token, tree_off, N, u_accept,
                                u_bonus, out=None, ws=None, stream=None):
    """Temperature-1 tree acceptance by rejection sampling with the caller's
    uniforms (fp64 [total_nodes] each).  Returns (accept_len, path, bonus)."""
    lib = load()
    _need(target_logits, "target_logits", torch.float32)
    _need(draft_logits, "draft_logits", torch.float32)
    for t, n in ((parent, "parent"), (token, "token"), (tree_off, "tree_off")):
        _need(t, n, torch.int32)
    _need(u_accept, "u_accept", torch.float64)
    _need(u_bonus, "u_bonus", torch.float64)
    total, V = target_logits.shape
    nseq = tree_off.numel() - 1
    dev = target_logits.device
    if out is None:
        out = (torch.empty(nseq, dtype=torch.int32, device=dev),
               torch.empty((nseq, N + 1), dtype=torch.int32, device=dev),
               torch.empty(nseq, dtype=torch.int32, device=dev))
    acc, path, bonus = out
    if ws is None:
        ws = workspace(jt_workspace_size(JT_OP_VERIFY_ACCEPT, nseq, 0, 0, 0, total), dev)
    rc = lib.jt_verify_accept_stochastic(_ptr(target_logits), _ptr(draft_logits), _ptr(parent), _ptr(token),
                                         _ptr(tree_off), nseq, N, V, total, _ptr(u_accept), _ptr(u_bonus),
                                         _ptr(acc), _ptr(path), _ptr(bonus), _ptr(ws), ws.numel(),
                                         _stream(stream))
    _check(rc, "jt_verify_accept_stochastic")
    return acc, path, bonus


@_on_tensor_device
def jt_check(ws: torch.Tensor, stream=None) -> None:
    """Synchronise and raise if a kernel flagged a device-side error in ws."""
    _check(load().jt_check(_ptr(ws), _stream(stream)), "jt_check")


@_on_tensor_device
def jt_tree_build(draft_logits, root_token, tree_off, W, total_nodes=None, out=None, ws=None,
                  stream=None):
    """Best-first draft tree from per-depth draft logits [nseq, N, V] (fp32).

    Returns (parent, token, depth, anc) on the device."""
    lib = load()
    _need(draft_logits, "draft_logits", torch.float32)
    _need(root_token, "root_token", torch.int32)
    _need(tree_off, "tree_off", torch.int32)
    nseq, N, V = draft_logits.shape
    if total_nodes is None:
        total_nodes = int(tree_off[-1].item())
    dev = draft_logits.device
    if out is None:
        out = (torch.empty(total_nodes, dtype=torch.int32, device=dev),
               torch.empty(total_nodes, dtype=torch.int32, device=dev),
               torch.empty(total_nodes, dtype=torch.int32, device=dev),
               torch.empty((total_nodes, 8), dtype=torch.int32, device=dev))
    parent, token, depth, anc = out
    if ws is None:
        ws = workspace(jt_workspace_size(JT_OP_TREE_BUILD, nseq, N, W, V), dev)
    rc = lib.jt_tree_build(_ptr(draft_logits), _ptr(root_token), _ptr(tree_off), nseq, N, W, V,
                           total_nodes, _ptr(parent), _ptr(token), _ptr(depth), _ptr(anc),
                           _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "jt_tree_build")
    return parent, token, depth, anc


@_on_tensor_device
def jt_tree_build_mixed(draft_logits, root_token, tree_off, W, alpha, total_nodes=None, out=None, ws=None,
                        stream=None):
    """jt_tree_build whose step scores are (1 - alpha) * log-prob - alpha *
    entropy(draft row), alpha in [0, 1] (1: pure entropy score).

    Returns (parent, token, depth, anc) on the device."""
    lib = load()
    _need(draft_logits, "draft_logits", torch.float32)
    _need(root_token, "root_token", torch.int32)
    _need(tree_off, "tree_off", torch.int32)
    nseq, N, V = draft_logits.shape
    if total_nodes is None:
        total_nodes = int(tree_off[-1].item())
    dev = draft_logits.device
    if out is None:
        out = (torch.empty(total_nodes, dtype=torch.int32, device=dev),
               torch.empty(total_nodes, dtype=torch.int32, device=dev),
               torch.empty(total_nodes, dtype=torch.int32, device=dev),
               torch.empty((total_nodes, 8), dtype=torch.int32, device=dev))
    parent, token, depth, anc = out
    if ws is None:
        ws = workspace(jt_workspace_size(JT_OP_TREE_BUILD_MIXED, nseq, N, W, V), dev)
    rc = lib.jt_tree_build_mixed(_ptr(draft_logits), _ptr(root_token), _ptr(tree_off), nseq, N, W, V,
                                 total_nodes, float(alpha), _ptr(parent), _ptr(token), _ptr(depth),
                                 _ptr(anc), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "jt_tree_build_mixed")
    return parent, token, depth, anc


@_on_tensor_device
def jt_tree_build_noalloc(draft_logits, root_token, tree_off, W, total_nodes=None, out=None,
                          sync_check=True, stream=None):
    """jt_tree_build with the library's fixed device scratch instead of a
    workspace (no allocation inside the library; the output tensors are the
    caller's).  Calls whose executions overlap on one device race on that
    scratch.  Returns (parent, token, depth, anc) on the device."""
    lib = load()
    _need(draft_logits, "draft_logits", torch.float32)
    _need(root_token, "root_token", torch.int32)
    _need(tree_off, "tree_off", torch.int32)
    nseq, N, V = draft_logits.shape
    if total_nodes is None:
        total_nodes = int(tree_off[-1].item())
    dev = draft_logits.device
    if out is None:
        out = (torch.empty(total_nodes, dtype=torch.int32, device=dev),
               torch.empty(total_nodes, dtype=torch.int32, device=dev),
               torch.empty(total_nodes, dtype=torch.int32, device=dev),
               torch.empty((total_nodes, 8), dtype=torch.int32, device=dev))
    parent, token, depth, anc = out
    rc = lib.jt_tree_build_noalloc(_ptr(draft_logits), _ptr(root_token), _ptr(tree_off), nseq, N, W,
                                   V, total_nodes, _ptr(parent), _ptr(token), _ptr(depth), _ptr(anc),
                                   1 if sync_check else 0, _stream(stream))
    _check(rc, "jt_tree_build_noalloc")
    return parent, token, depth, anc


@_on_tensor_device
def jt_tree_topw(logits, W, ws=None, stream=None):
    """Top-W ids (int32), log-probs and lse (fp64) of every row of [..., V] fp32."""
    lib = load()
    _need(logits, "logits", torch.float32)
    V = logits.shape[-1]
    rows = logits.numel() // V
    dev = logits.device
    tok = torch.empty(logits.shape[:-1] + (W,), dtype=torch.int32, device=dev)
    lp = torch.empty(logits.shape[:-1] + (W,), dtype=torch.float64, device=dev)
    lse = torch.empty(logits.shape[:-1], dtype=torch.float64, device=dev)
    if ws is None:
        ws = workspace(jt_workspace_size(JT_OP_TREE_TOPW, rows, 1, W, V), dev)
    rc = lib.jt_tree_topw(_ptr(logits), rows, V, W, _ptr(tok), _ptr(lp), _ptr(lse), _ptr(ws),
                          ws.numel(), _stream(stream))
    _check(rc, "jt_tree_topw")
    return tok, lp, lse


@_on_tensor_device
def jt_tree_expand(tok, lp, root_token, tree_off, total_nodes=None, ws=None, stream=None):
    """Best-first expansion from given tables tok [nseq,N,W] int32, lp fp64."""
    lib = load()
    _need(tok, "tok", torch.int32)
    _need(lp, "lp", torch.float64)
    _need(root_token, "root_token", torch.int32)
    _need(tree_off, "tree_off", torch.int32)
    nseq, N, W = tok.shape
    if total_nodes is None:
        total_nodes = int(tree_off[-1].item())
    dev = tok.device
    parent = torch.empty(total_nodes, dtype=torch.int32, device=dev)
    token = torch.empty_like(parent)
    depth = torch.empty_like(parent)
    anc = torch.empty((total_nodes, 8), dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(256, dev)
    rc = lib.jt_tree_expand(_ptr(tok), _ptr(lp), _ptr(root_token), _ptr(tree_off), nseq, N, W,
                            total_nodes, _ptr(parent), _ptr(token), _ptr(depth), _ptr(anc),
                            _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "jt_tree_expand")
    return parent, token, depth, anc


@_on_tensor_device
def jt_tree_expand_capped(tok, lp, root_token, tree_off, w_cap=None, n_cap=None, total_nodes=None, ws=None,
                          stream=None):
    """jt_tree_expand with optional per-sequence width / depth caps
    (int32 [nseq] device tensors)."""
    lib = load()
    _need(tok, "tok", torch.int32)
    _need(lp, "lp", torch.float64)
    _need(root_token, "root_token", torch.int32)
    _need(tree_off, "tree_off", torch.int32)
    for t, name in ((w_cap, "w_cap"), (n_cap, "n_cap")):
        if t is not None:
            _need(t, name, torch.int32)
    nseq, N, W = tok.shape
    if total_nodes is None:
        total_nodes = int(tree_off[-1].item())
    dev = tok.device
    parent = torch.empty(total_nodes, dtype=torch.int32, device=dev)
    token = torch.empty_like(parent)
    depth = torch.empty_like(parent)
    anc = torch.empty((total_nodes, 8), dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(256, dev)
    rc = lib.jt_tree_expand_capped(_ptr(tok), _ptr(lp), _ptr(root_token), _ptr(tree_off), _ptr(w_cap),
                                   _ptr(n_cap), nseq, N, W, total_nodes, _ptr(parent), _ptr(token),
                                   _ptr(depth), _ptr(anc), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "jt_tree_expand_capped")
    return parent, token, depth, anc


@_on_tensor_device
def jt_tree_policy(lp, accept_len, budget_state, acc_ema, params=None, out=None, ws=None, stream=None):
    """One step of the adaptive tree policy.  lp fp64 [nseq, N, W];
    accept_len int32 [nseq] or None; budget_state int32 / acc_ema fp64
    [nseq] are updated in place.  Returns (tree_off, w_cap, n_cap)."""
    lib = load()
    _need(lp, "lp", torch.float64)
    _need(budget_state, "budget_state", torch.int32)
    _need(acc_ema, "acc_ema", torch.float64)
    if accept_len is not None:
        _need(accept_len, "accept_len", torch.int32)
    nseq, N, W = lp.shape
    params = params or policy_params()
    dev = lp.device
    if out is None:
        out = (torch.empty(nseq + 1, dtype=torch.int32, device=dev),
               torch.empty(nseq, dtype=torch.int32, device=dev),
               torch.empty(nseq, dtype=torch.int32, device=dev))
    tree_off, w_cap, n_cap = out
    if ws is None:
        ws = workspace(jt_workspace_size(JT_OP_TREE_POLICY), dev)
    rc = lib.jt_tree_policy(_ptr(lp), nseq, N, W, _ptr(accept_len), ctypes.byref(params), _ptr(budget_state),
                            _ptr(acc_ema), _ptr(tree_off), _ptr(w_cap), _ptr(n_cap), _ptr(ws), ws.numel(),
                            _stream(stream))
    _check(rc, "jt_tree_policy")
    return tree_off, w_cap, n_cap


@_on_tensor_device
def jt_tree_build_adaptive(draft_logits, root_token, accept_len, budget_state, acc_ema, W, params=None,
                           capacity=None, out=None, ws=None, stream=None):
    """Top-W tables, adaptive policy and capped expansion in one call.
    Returns (tree_off, w_cap, n_cap, parent, token, depth, anc); the node
    arrays have `capacity` rows (default nseq * the policy's ceiling)."""
    lib = load()
    _need(draft_logits, "draft_logits", torch.float32)
    _need(root_token, "root_token", torch.int32)
    _need(budget_state, "budget_state", torch.int32)
    _need(acc_ema, "acc_ema", torch.float64)
    if accept_len is not None:
        _need(accept_len, "accept_len", torch.int32)
    nseq, N, V = draft_logits.shape
    params = params or policy_params()
    if capacity is None:
        capacity = nseq * policy_ceiling(params, nseq)
    dev = draft_logits.device
    if out is None:
        out = (torch.empty(nseq + 1, dtype=torch.int32, device=dev),
               torch.empty(nseq, dtype=torch.int32, device=dev),
               torch.empty(nseq, dtype=torch.int32, device=dev),
               torch.empty(capacity, dtype=torch.int32, device=dev),
               torch.empty(capacity, dtype=torch.int32, device=dev),
               torch.empty(capacity, dtype=torch.int32, device=dev),
               torch.empty((capacity, 8), dtype=torch.int32, device=dev))
    tree_off, w_cap, n_cap, parent, token, depth, anc = out
    if ws is None:
        ws = workspace(jt_workspace_size(JT_OP_TREE_BUILD, nseq, N, W, V), dev)
    rc = lib.jt_tree_build_adaptive(_ptr(draft_logits), _ptr(root_token), nseq, N, W, V, capacity,
                                    _ptr(accept_len), ctypes.byref(params), _ptr(budget_state), _ptr(acc_ema),
                                    _ptr(tree_off), _ptr(w_cap), _ptr(n_cap), _ptr(parent), _ptr(token),
                                    _ptr(depth), _ptr(anc), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "jt_tree_build_adaptive")
    return tree_off, w_cap, n_cap, parent, token, depth, anc


@_on_tensor_device
def jt_tree_attn_paged(q, k_cache, v_cache, block_table, prefix_len, tree_off, anc, scale=None,
                       max_tree=None, out=None, lse=None, ws=None, stream=None, with_lse=True):
    """Tree-causal attention over a paged KV cache.

    q [total, Hq, D]; k/v [pages, 16, Hkv, D] (both bf16, or both fp32);
    block_table [nseq, max_pages] int32; prefix_len [nseq] int32;
    tree_off [nseq+1] int32; anc [total, 8] int32/uint32 ancestor sets.
    Returns (out, lse)."""
    lib = load()
    if q.dtype == torch.bfloat16:
        dtype = JT_DTYPE_BF16
    elif q.dtype == torch.float32:
        dtype = JT_DTYPE_F32
    else:
        raise TypeError("q must be bf16 or fp32")
    _need(q, "q", None)
    _need(k_cache, "k_cache", q.dtype)
    _need(v_cache, "v_cache", q.dtype)
    _need(block_table, "block_table", torch.int32)
    _need(prefix_len, "prefix_len", torch.int32)
    _need(tree_off, "tree_off", torch.int32)
    _need(anc, "anc", None)
    total, Hq, D = q.shape
    num_pages, page, Hkv, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("q and k_cache head dims differ")
    nseq, max_pages = block_table.shape
    if max_tree is None:
        max_tree = int((tree_off[1:] - tree_off[:-1]).max().item())
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((total, Hq), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(jt_workspace_size(JT_OP_TREE_ATTN, nseq, 0, 0, 0, total, Hq, Hkv, D,
                                         max_pages, max_tree), q.device)
    rc = lib.jt_tree_attn_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), dtype, _ptr(block_table),
                                max_pages, num_pages, _ptr(prefix_len), _ptr(tree_off), _ptr(anc),
                                nseq, total, max_tree, Hq, Hkv, D, page, float(scale), _ptr(out),
                                _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "jt_tree_attn_paged")
    return out, lse


@_on_tensor_device
def jt_verify_accept(target_logits, parent, token, tree_off, N, rule=JT_RULE_GREEDY, t=None,
                     log_t=None, out=None, ws=None, stream=None):
    """Tree acceptance: returns (accept_len [nseq], path [nseq, N+1], bonus [nseq])."""
    lib = load()
    _need(target_logits, "target_logits", torch.float32)
    _need(parent, "parent", torch.int32)
    _need(token, "token", torch.int32)
    _need(tree_off, "tree_off", torch.int32)
    total, V = target_logits.shape
    nseq = tree_off.numel() - 1
    if isinstance(rule, str):
        rule = {"greedy": JT_RULE_GREEDY, "margin": JT_RULE_MARGIN}[rule]
    if log_t is None:
        log_t = math.log(t) if t is not None else 0.0
    dev = target_logits.device
    if out is None:
        out = (torch.empty(nseq, dtype=torch.int32, device=dev),
               torch.empty((nseq, N + 1), dtype=torch.int32, device=dev),
               torch.empty(nseq, dtype=torch.int32, device=dev))
    acc, path, bonus = out
    if ws is None:
        ws = workspace(jt_workspace_size(JT_OP_VERIFY_ACCEPT, nseq, 0, 0, 0, total), dev)
    rc = lib.jt_verify_accept(_ptr(target_logits), _ptr(parent), _ptr(token), _ptr(tree_off), nseq,
                              N, V, total, rule, float(log_t), _ptr(acc), _ptr(path), _ptr(bonus),
                              _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "jt_verify_accept")
    return acc, path, bonus


@_on_tensor_device
def jt_selftest_wait_timeout(ws=None, stream=None):
    """Run the bounded-wait timeout diagnostic; returns the workspace whose
    error word it sets (read it with jt_check: JT_ERR_TIMEOUT)."""
    lib = load()
    if ws is None:
        ws = workspace(256)
    _check(lib.jt_selftest_wait_timeout(_ptr(ws), ws.numel(), _stream(stream)), "jt_selftest_wait_timeout")
    return ws
