"""GPU parity of the tree build (jt_tree_topw / jt_tree_expand /
jt_tree_build) against the oracle: bit-exact integers, lse within 1e-9.

Layered as follows: top-W ids must match exactly (pure fp32 compares);
lse within 1e-9 absolute; the expansion fed the oracle's own tables must be
bit-exact; the end-to-end tree must be bit-exact unless the oracle reports a
decision gap below 1e-9 (a near-tie that rounding could flip), which would
be reported as ambiguous rather than passed."""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_jt_gb300 as jt
from tree_speculative_decoding_jt_gb300 import workloads as wk
from gpu_util import dev

pytestmark = pytest.mark.gpu

AMBIGUOUS_GAP = 1e-9


@pytest.mark.parametrize("V,W,rows", [(1000, 2, 4), (151936, 4, 6), (4099, 8, 5), (1001, 3, 3),
                                      (5, 5, 2), (8192, 1, 3)])
def test_topw_lse_matches_oracle(V, W, rows):
    rng = np.random.default_rng(V + W)
    z = (rng.standard_normal((rows, V)) * np.sqrt(2)).astype(np.float32)
    z[0, 7 % V] = z[0, 3 % V] = z[0].max() + 0.5       # tie on the maximum
    if rows > 2:
        z[2, :] = -np.inf
        z[2, V // 2] = 1.0
    tok, lp, lse = jt.jt_tree_topw(dev(z), W)
    torch.cuda.synchronize()
    otok, olp, olse = oracle.topw_lse(z, W)
    np.testing.assert_array_equal(tok.cpu().numpy(), otok)
    d = np.abs(lse.cpu().numpy() - olse)
    assert d.max() <= 1e-9, d
    got_lp = lp.cpu().numpy()
    fin = np.isfinite(olp)
    np.testing.assert_array_equal(np.isfinite(got_lp), fin)  # -inf (probability 0) on the same entries
    dl = np.abs(got_lp[fin] - olp[fin])
    assert dl.max() <= 1e-9


def _expand_case(seed, nseq, N, W, budgets, ties=False):
    rng = np.random.default_rng(seed)
    lp = -np.sort(rng.exponential(1.0, size=(nseq, N, W)), axis=2)
    if ties:
        lp = np.round(lp, 1)
    tok = np.stack([np.stack([np.sort(rng.choice(1000, size=W, replace=False)) for _ in range(N)])
                    for _ in range(nseq)]).astype(np.int32)
    root = rng.integers(0, 1000, size=nseq).astype(np.int32)
    off = np.concatenate([[0], np.cumsum(budgets)]).astype(np.int32)
    return tok, lp, root, off


@pytest.mark.parametrize("N,W,budgets,ties", [
    (4, 2, [16, 1, 31], False), (16, 4, [256, 128, 7], False), (5, 3, [200, 64], True),
    (16, 1, [17, 2], False), (6, 8, [256, 255, 9], True), (2, 4, [21, 5], False)])
def test_expand_bit_exact_from_oracle_tables(N, W, budgets, ties):
    tok, lp, root, off = _expand_case(N * 100 + W, len(budgets), N, W, budgets, ties)
    want = oracle.tree_expand(tok, lp, root, off, N, W)
    par, tk, dp, anc = jt.jt_tree_expand(dev(tok), dev(lp), dev(root), dev(off), int(off[-1]))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(par.cpu().numpy(), want["parent"])
    np.testing.assert_array_equal(tk.cpu().numpy(), want["token"])
    np.testing.assert_array_equal(dp.cpu().numpy(), want["depth"])
    np.testing.assert_array_equal(anc.cpu().numpy().view(np.uint32), want["anc"])


def _build_and_compare(wl):
    want = oracle.tree_build(wl.draft_logits, wl.root_token, wl.tree_off, wl.cfg["W"])
    if np.min(want["gap"]) < AMBIGUOUS_GAP:
        pytest.skip(f"ambiguous: oracle decision gap {np.min(want['gap']):.3g} below rounding noise")
    out = jt.jt_tree_build(dev(wl.draft_logits), dev(wl.root_token), dev(wl.tree_off),
                           wl.cfg["W"], total_nodes=wl.total)
    torch.cuda.synchronize()
    par, tk, dp, anc = (t.cpu().numpy() for t in out)
    np.testing.assert_array_equal(par, want["parent"])
    np.testing.assert_array_equal(tk, want["token"])
    np.testing.assert_array_equal(dp, want["depth"])
    np.testing.assert_array_equal(anc.view(np.uint32), want["anc"])
    return want


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_build_bit_exact_full_configs(cfg):
    wl = wk.make(cfg, with_draft=True, with_kv=False)
    _build_and_compare(wl)


@pytest.mark.parametrize("seed", range(6))
def test_build_bit_exact_ragged_small(seed):
    rng = np.random.default_rng(seed)
    nseq = int(rng.integers(1, 9))
    N, W = int(rng.integers(1, 9)), int(rng.integers(1, 9))
    full = sum(W ** d for d in range(N + 1))
    budgets = tuple(int(rng.integers(1, min(full, 256) + 1)) for _ in range(nseq))
    o = dict(dtype="f32", nseq=nseq, Hq=4, Hkv=1, D=64, prefix=("fixed", 16), budgets=budgets,
             N=N, W=W, V=int(rng.integers(W, 3000)), qkv_std=1.0)
    _build_and_compare(wk.make(1, seed=seed, overrides=o))


def test_build_budget_beyond_full_tree_flags_error():
    z = dev(np.zeros((2, 2, 10), np.float32))
    off = dev(np.array([0, 7, 15], np.int32))   # second tree: 8 > 1 + 2 + 4
    ws = jt.workspace(jt.jt_workspace_size(jt.JT_OP_TREE_BUILD, 2, 2, 2, 10))
    jt.jt_tree_build(z, dev(np.array([1, 2], np.int32)), off, 2, total_nodes=15, ws=ws)
    with pytest.raises(jt.JtError) as e:
        jt.jt_check(ws)
    assert e.value.status == -1
    jt.jt_check(ws)  # cleared


def test_build_host_side_argument_errors():
    z = dev(np.zeros((1, 2, 10), np.float32))
    off = dev(np.array([0, 3], np.int32))
    with pytest.raises(jt.JtError):
        jt.jt_tree_build(z, dev(np.array([1], np.int32)), off, 9, total_nodes=3)  # W > 8
    with pytest.raises(jt.JtError) as e:
        jt.jt_tree_build(z, dev(np.array([1], np.int32)), off, 2, total_nodes=3, ws=jt.workspace(256))
    assert e.value.status == -5  # workspace too small


@pytest.mark.parametrize("N,W,budget,scale,depth", [(64, 1, 65, 1.4, 64), (64, 2, 256, 40.0, 64),
                                                    (64, 8, 256, 40.0, 60), (64, 8, 256, 0.05, 2)])
def test_build_bit_exact_maximum_depth_and_width(N, W, budget, scale, depth):
    """The build's limits: depth 64, width 8, budget 256.  Peaked rows (a
    large logit scale: the top-1 log-prob near 0) give trees about 64 deep;
    near-uniform rows give wide, shallow ones; W = 1 is the full chain of
    64 drafted nodes.  `depth`: the least deepest node the case reaches."""
    o = dict(dtype="f32", nseq=2, Hq=4, Hkv=1, D=64, prefix=("fixed", 0), budgets=(budget,), N=N, W=W,
             V=700, qkv_std=1.0)
    wl = wk.make(1, seed=N + W, overrides=o, with_kv=False)
    wl.draft_logits[:] *= np.float32(scale / np.sqrt(2))
    want = _build_and_compare(wl)
    assert want["depth"].max() >= depth
