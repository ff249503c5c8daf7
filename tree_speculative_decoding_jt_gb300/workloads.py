"""Seeded synthetic inputs for the tree speculative decoding hot path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no top-W, no softmax, no acceptance).  Both the CUDA path
(tests, bench) and the CPU oracle are fed from here, so the two sides always
see identical inputs.

The workloads mirror the shapes of the pages' setting (a Qwen3-8B-shaped
attention layer: 32 query heads, 8 KV heads, head dim 128, bf16, vocab
151936, paged KV with 16-token pages) with values drawn from fixed
distributions.  No model weights or benchmark data are involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PAGE_SIZE = 16

# name, dtype, nseq, Hq, Hkv, D, prefix rule, tree budgets, N, W, V,
# q/k/v std, target boost, boosted fraction.
CONFIGS = {
    1: dict(name="tiny-f32-L128-B16", dtype="f32", nseq=1, Hq=4, Hkv=1, D=64,
            prefix=("fixed", 128), budgets=(16,), N=4, W=2, V=1000, qkv_std=1.0,
            boost=3.0, boost_frac=0.7, t=0.8),
    2: dict(name="qwen3-8b-attn-b1-L4096-B256", dtype="bf16", nseq=1, Hq=32, Hkv=8, D=128,
            prefix=("fixed", 4096), budgets=(256,), N=16, W=4, V=151936, qkv_std=0.5,
            boost=4.0, boost_frac=0.8, t=0.8),
    3: dict(name="serving-b16-L1k-8k-B128-256", dtype="bf16", nseq=16, Hq=32, Hkv=8, D=128,
            prefix=("uniform", 1024, 8192), budgets=(128,) * 8 + (256,) * 8, N=16, W=4,
            V=151936, qkv_std=0.5, boost=4.0, boost_frac=0.8, t=0.8),
    4: dict(name="long-b32-L32768-B64", dtype="bf16", nseq=32, Hq=32, Hkv=8, D=128,
            prefix=("fixed", 32768), budgets=(64,), N=8, W=4, V=151936, qkv_std=0.5,
            boost=4.0, boost_frac=0.8, t=0.8),
    5: dict(name="verify-step-b8-L2k-16k-B256", dtype="bf16", nseq=8, Hq=32, Hkv=8, D=128,
            prefix=("uniform", 2048, 16384), budgets=(256,), N=16, W=4, V=151936,
            qkv_std=0.5, boost=4.0, boost_frac=0.8, t=0.8),
    # the drafter's own tree forward: a draft head with the target layer's
    # attention shape attends among the tree nodes only (no prefix slots)
    6: dict(name="drafter-tree-b16-L0-B256", dtype="bf16", nseq=16, Hq=32, Hkv=8, D=128,
            prefix=("fixed", 0), budgets=(256,), N=16, W=4, V=151936,
            qkv_std=0.5, boost=4.0, boost_frac=0.8, t=0.8),
}

DRAFT_STD = math.sqrt(2.0)   # "N(0,2)": variance 2
TARGET_STD = math.sqrt(2.0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    cfg: dict
    seed: int
    draft_logits: np.ndarray      # [nseq, N, V] float32
    root_token: np.ndarray        # [nseq] int32
    tree_off: np.ndarray          # [nseq+1] int32, B_b = tree_off[b+1]-tree_off[b]
    prefix_len: np.ndarray        # [nseq] int32
    block_table: np.ndarray       # [nseq, max_pages] int32, -1 where unused
    k_cache: np.ndarray           # [pages, 16, Hkv, D] float32 or uint16 (bf16 bits)
    v_cache: np.ndarray
    q: np.ndarray                 # [total, Hq, D] float32 or uint16 (bf16 bits)
    scale: float
    guard_pages: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))

    @property
    def nseq(self):
        return len(self.root_token)

    @property
    def total(self):
        return int(self.tree_off[-1])


def _normal(rng, shape, std):
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def make(cfg_id=None, seed=None, *, overrides=None, poison=False, n_guard=2,
         with_draft=True, with_kv=True) -> Workload:
    """Draw one workload.

    cfg_id: 1..5 picks a preset from CONFIGS; overrides replaces any preset
    field (e.g. smaller V or prefix for oracle-sized parity cases).  seed
    defaults to 1000 + cfg_id.  poison=True fills spare pool pages and the
    unused tail of every sequence's last page with NaN, so any read outside
    the block table or past the tree shows up in the output.  with_kv=False
    skips drawing q, K and V (they come last from the generator, so every
    other field is unchanged) for cases that only need the draft side.
    """
    cfg = dict(CONFIGS[cfg_id]) if cfg_id is not None else {}
    if overrides:
        cfg.update(overrides)
    if seed is None:
        seed = 1000 + (cfg_id or 0)
    rng = np.random.default_rng(seed)
    nseq, N, W, V = cfg["nseq"], cfg["N"], cfg["W"], cfg["V"]
    Hq, Hkv, D = cfg["Hq"], cfg["Hkv"], cfg["D"]
    page = cfg.get("page_size", PAGE_SIZE)

    budgets = list(cfg["budgets"])
    if len(budgets) == 1:
        budgets = budgets * nseq
    assert len(budgets) == nseq
    tree_off = np.zeros(nseq + 1, np.int32)
    tree_off[1:] = np.cumsum(budgets)

    pr = cfg["prefix"]
    if pr[0] == "fixed":
        prefix_len = np.full(nseq, pr[1], np.int32)
    elif pr[0] == "uniform":
        prefix_len = rng.integers(pr[1], pr[2] + 1, size=nseq).astype(np.int32)
    elif pr[0] == "list":
        prefix_len = np.asarray(pr[1], np.int32)
    else:
        raise ValueError(pr)

    # paged pool: pages for prefix + tree of every sequence, plus guard pages,
    # physical ids randomly permuted over the pool
    need = [(int(prefix_len[b]) + budgets[b] + page - 1) // page for b in range(nseq)]
    max_pages = max(need)
    n_pages = sum(need) + n_guard
    perm = rng.permutation(n_pages).astype(np.int32)
    block_table = np.full((nseq, max_pages), -1, np.int32)
    pos = 0
    for b in range(nseq):
        block_table[b, :need[b]] = perm[pos:pos + need[b]]
        pos += need[b]
    guard = perm[pos:]

    draft = _normal(rng, (nseq, N, V), DRAFT_STD) if with_draft else None
    root_token = rng.integers(0, V, size=nseq).astype(np.int32)

    if not with_kv:
        return Workload(cfg=cfg, seed=seed, draft_logits=draft, root_token=root_token,
                        tree_off=tree_off, prefix_len=prefix_len, block_table=block_table,
                        k_cache=None, v_cache=None, q=None, scale=1.0 / math.sqrt(D), guard_pages=guard)
    std = cfg["qkv_std"]
    total = int(tree_off[-1])
    kf = _normal(rng, (n_pages, page, Hkv, D), std)
    vf = _normal(rng, (n_pages, page, Hkv, D), std)
    qf = _normal(rng, (total, Hq, D), std)
    if cfg.get("q_mult"):
        qf *= np.float32(cfg["q_mult"])
    if poison:
        for arr in (kf, vf):
            arr[guard] = np.nan
            for b in range(nseq):
                used = int(prefix_len[b]) + budgets[b]
                last = block_table[b, need[b] - 1]
                off = used - (need[b] - 1) * page
                arr[last, off:] = np.nan
    if cfg["dtype"] == "bf16":
        k, v, q = f32_to_bf16_bits(kf), f32_to_bf16_bits(vf), f32_to_bf16_bits(qf)
    else:
        k, v, q = kf, vf, qf
    return Workload(cfg=cfg, seed=seed, draft_logits=draft, root_token=root_token,
                    tree_off=tree_off, prefix_len=prefix_len, block_table=block_table,
                    k_cache=k, v_cache=v, q=q, scale=1.0 / math.sqrt(D), guard_pages=guard)


def target_logits(wl: Workload, parent: np.ndarray, token: np.ndarray, *, seed=None,
                  boost=None, frac=None, deep=False) -> np.ndarray:
    """Target logits [total, V] ~ N(0,2) for a built tree.

    For each non-root node c, with probability ``frac`` the drafted token is
    boosted in the row that verifies it (the row of c's parent): by
    ``+boost``, or, with deep=True, set to that row's largest value plus
    ``boost`` so that long accepted paths occur."""
    cfg = wl.cfg
    V = cfg["V"]
    boost = cfg["boost"] if boost is None else boost
    frac = cfg["boost_frac"] if frac is None else frac
    rng = np.random.default_rng((wl.seed * 7919 + 17) if seed is None else seed)
    total = wl.total
    z = _normal(rng, (total, V), TARGET_STD)
    hit = rng.random(total) < frac
    for b in range(wl.nseq):
        off, end = int(wl.tree_off[b]), int(wl.tree_off[b + 1])
        for c in range(off + 1, end):
            if not hit[c]:
                continue
            row = off + int(parent[c])
            t = int(token[c])
            if deep:
                z[row, t] = z[row].max() + np.float32(boost)
            else:
                z[row, t] += np.float32(boost)
    return z
