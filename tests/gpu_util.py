"""Helpers shared by the GPU tests: move seeded workloads to the device and
compare with the oracle."""
import numpy as np
import torch

import oracle
from tree_speculative_decoding_jt_gb300 import workloads as wk


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_np_bf16(t):
    return wk.bf16_bits_to_f32(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))


def kv_to_device(wl):
    if wl.q.dtype == np.uint16:
        return dev_bf16(wl.q), dev_bf16(wl.k_cache), dev_bf16(wl.v_cache)
    return dev(wl.q), dev(wl.k_cache), dev(wl.v_cache)


def oracle_tree(wl):
    """Tree of a workload built by the oracle (the CUDA path never supplies
    oracle inputs)."""
    return oracle.tree_build(wl.draft_logits, wl.root_token, wl.tree_off, wl.cfg["W"])


def attn_errors(got, want):
    d = np.abs(got.astype(np.float64) - want)
    return float(d.max()), float(d.mean())


def oracle_attn_threaded(wl, parent, rows, threads=None):
    """The oracle's attention for the nodes in `rows`, spread over host
    threads in contiguous chunks (the C oracle runs outside the interpreter
    lock); returns (out, lse) in the order of `rows`."""
    import concurrent.futures
    import os

    rows = np.asarray(rows, np.int32)
    if threads is None:
        try:
            threads = len(os.sched_getaffinity(0))
        except AttributeError:
            threads = os.cpu_count() or 1
    chunks = [c for c in np.array_split(rows, max(1, min(threads, len(rows)))) if len(c)]

    def one(c):
        return oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.prefix_len, wl.tree_off,
                                parent, wl.scale, rows=c)

    with concurrent.futures.ThreadPoolExecutor(len(chunks)) as ex:
        parts = list(ex.map(one, chunks))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])
