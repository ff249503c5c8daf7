"""The debug library variant (JT_LIB_VARIANT=checks: libjt built with
-DJT_CHECKS): device-side checks of input contents report JT_ERR_INVALID
through jt_check instead of computing on bad data.  Skipped unless the
process loads that variant (the default build compiles the checks out)."""
import math

import numpy as np
import pytest
import torch

import tree_speculative_decoding_jt_gb300 as jt
from tree_speculative_decoding_jt_gb300 import workloads as wk
from gpu_util import dev, kv_to_device, oracle_tree

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(jt.library_variant() != "checks", reason="needs JT_LIB_VARIANT=checks")]


def _small():
    o = dict(dtype="bf16", nseq=2, Hq=32, Hkv=8, D=128, prefix=("list", [300, 40]), budgets=(40, 17),
             N=5, W=3, V=300, qkv_std=0.5)
    return wk.make(2, seed=77, overrides=o)


def _attn(wl, bt, anc):
    q, k, v = kv_to_device(wl)
    ws = jt.workspace(jt.jt_workspace_size(jt.JT_OP_TREE_ATTN, wl.nseq, 0, 0, 0, wl.total, 32, 8, 128,
                                           bt.shape[1], 40))
    jt.jt_tree_attn_paged(q, k, v, dev(bt), dev(wl.prefix_len), dev(wl.tree_off), dev(anc.view(np.int32)),
                          scale=wl.scale, max_tree=40, ws=ws)
    return ws


def test_clean_inputs_pass_the_checks():
    wl = _small()
    ws = _attn(wl, wl.block_table, oracle_tree(wl)["anc"])
    jt.jt_check(ws)


def test_block_table_entry_outside_the_pool_is_flagged():
    wl = _small()
    bt = wl.block_table.copy()
    bt[0, 3] = wl.k_cache.shape[0] + 5   # past the pool: the copy reads fill values, the check flags it
    ws = _attn(wl, bt, oracle_tree(wl)["anc"])
    with pytest.raises(jt.JtError) as e:
        jt.jt_check(ws)
    assert e.value.status == jt.JT_ERR_INVALID


def test_ancestor_set_without_its_own_node_is_flagged():
    wl = _small()
    anc = oracle_tree(wl)["anc"].copy()
    anc[5, 0] &= ~np.uint32(1 << 5)      # node 5 of sequence 0 loses its own bit
    ws = _attn(wl, wl.block_table, anc)
    with pytest.raises(jt.JtError):
        jt.jt_check(ws)


def test_nan_target_logit_is_flagged_by_the_acceptance():
    wl = _small()
    tree = oracle_tree(wl)
    z = wk.target_logits(wl, tree["parent"], tree["token"])
    z[0, 17] = np.nan                    # the root row is always read
    ws = jt.workspace(jt.jt_workspace_size(jt.JT_OP_VERIFY_ACCEPT, wl.nseq, 0, 0, 0, wl.total))
    jt.jt_verify_accept(dev(z), dev(tree["parent"]), dev(tree["token"]), dev(wl.tree_off), wl.cfg["N"],
                        rule=jt.JT_RULE_MARGIN, log_t=math.log(0.8), ws=ws)
    with pytest.raises(jt.JtError):
        jt.jt_check(ws)


def test_nan_draft_logit_is_flagged_by_the_build():
    wl = _small()
    d = wl.draft_logits.copy()
    d[1, 2, 7] = np.nan
    ws = jt.workspace(jt.jt_workspace_size(jt.JT_OP_TREE_BUILD, wl.nseq, wl.cfg["N"], 3, wl.cfg["V"]))
    jt.jt_tree_build(dev(d), dev(wl.root_token), dev(wl.tree_off), 3, total_nodes=wl.total, ws=ws)
    with pytest.raises(jt.JtError):
        jt.jt_check(ws)
    torch.cuda.synchronize()
