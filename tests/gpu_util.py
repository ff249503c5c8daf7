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
