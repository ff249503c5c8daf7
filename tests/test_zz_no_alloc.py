"""jt_tree_build_noalloc (the build with the library's fixed device scratch)
against jt_tree_build (caller workspace): identical trees on two calls in a
row, and a refusal, before any device work, of a build whose tables do not
fit the fixed scratch.

The file name sorts last so the GPU case also runs after every other test
has used the device."""
import ctypes

import numpy as np
import pytest
import torch

import tree_speculative_decoding_jt_gb300 as jt
from tree_speculative_decoding_jt_gb300 import workloads as wk

JT_ERR_WORKSPACE = -5
SCRATCH_BYTES = 4 * 1024 * 1024


def test_oversized_build_is_refused_on_the_host():
    lib = jt.load()
    nseq, N, W, V = 1024, 16, 4, 151936         # 16384 rows: well past 4 MiB of tables
    need = jt.jt_workspace_size(jt.JT_OP_TREE_BUILD, nseq, N, W, V)
    assert need > SCRATCH_BYTES
    fake = ctypes.c_void_p(4096)                  # never dereferenced: refused before any device work is enqueued
    rc = lib.jt_tree_build_noalloc(fake, fake, fake, nseq, N, W, V, nseq * 16, fake, fake, fake,
                                   fake, 1, None)
    assert rc == JT_ERR_WORKSPACE
    # the case size the scratch is documented to hold still passes the size check
    assert jt.jt_workspace_size(jt.JT_OP_TREE_BUILD, 256, 16, 4, 151936) <= SCRATCH_BYTES


@pytest.mark.gpu
def test_noalloc_matches_workspace_build_twice_in_a_row():
    dev = torch.device("cuda:0")
    for cfg, seed in ((2, 11), (3, 12)):       # two different shapes back to back
        wl = wk.make(cfg, seed=seed)
        z = torch.from_numpy(wl.draft_logits).to(dev)
        root = torch.from_numpy(wl.root_token).to(dev)
        off = torch.from_numpy(wl.tree_off).to(dev)
        W = wl.cfg["W"]
        want = [t.cpu().numpy() for t in jt.jt_tree_build(z, root, off, W, total_nodes=wl.total)]
        for _ in range(2):
            got = jt.jt_tree_build_noalloc(z, root, off, W, total_nodes=wl.total, sync_check=True)
            for g, w in zip(got, want):
                np.testing.assert_array_equal(g.cpu().numpy(), w)
    # the asynchronous form gives the same tree
    got = jt.jt_tree_build_noalloc(z, root, off, W, total_nodes=wl.total, sync_check=False)
    torch.cuda.synchronize()
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g.cpu().numpy(), w)
