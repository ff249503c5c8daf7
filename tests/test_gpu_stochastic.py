"""GPU parity of jt_verify_accept_stochastic against the oracle, with the
same seeded uniforms.  The kernel's softmax and sums are fp32, the
oracle's fp64, so decisions taken within rounding of their thresholds may
differ:
  * a sequence whose acceptance tests all lie further than 1e-4 from their
    thresholds must give the same accept_len and path (the oracle reports
    that margin); closer sequences are counted as ambiguous, their count is
    printed, and at most 5 % of a case's sequences may be ambiguous (with
    fewer than 20 sequences: none).  1e-4 bounds the kernel's fp32 error in
    min(1, r/q): a softmax over at most 151936 entries and a residual
    rewrite per rejection, each a few fp32 roundings relative;
  * its bonus must be a valid draw from the oracle's final residual r: the
    kernel's token x has r(x) > 0 and its CDF bin contains the uniform
    within 1e-4; when the uniform lies further than 1e-4 inside the
    oracle's own bin the two tokens must be equal."""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_jt_gb300 as jt
from tree_speculative_decoding_jt_gb300 import workloads as wk
from gpu_util import dev, oracle_tree

pytestmark = pytest.mark.gpu

MARGIN = 1e-4
CDF_TOL = 1e-4


MAX_AMBIGUOUS = 0.05


def _compare(target, draft, parent, token, off, N, ua, ub):
    want_acc, want_path, want_bonus, margin, fr, fu = oracle.verify_accept_stochastic(
        target, draft, parent, token, off, N, ua, ub, with_residual=True)
    acc, path, bonus = jt.jt_verify_accept_stochastic(dev(target), dev(draft), dev(parent), dev(token),
                                                      dev(off), N, dev(ua), dev(ub))
    torch.cuda.synchronize()
    acc, path, bonus = acc.cpu().numpy(), path.cpu().numpy(), bonus.cpu().numpy()
    clear = margin > MARGIN
    n_amb = int((~clear).sum())
    print(f"stochastic parity: {n_amb} of {len(clear)} sequences ambiguous (a test within {MARGIN} of its threshold)")
    assert n_amb <= int(MAX_AMBIGUOUS * len(clear)), f"{n_amb} of {len(clear)} sequences ambiguous"
    np.testing.assert_array_equal(acc[clear], want_acc[clear])
    np.testing.assert_array_equal(path[clear], want_path[clear])
    V = target.shape[1]
    assert np.all((bonus >= 0) & (bonus < V))
    exact = 0
    for b in np.nonzero(clear)[0]:
        cdf = np.cumsum(fr[b])
        x, xw, u = int(bonus[b]), int(want_bonus[b]), fu[b]
        lo = cdf[x - 1] if x > 0 else 0.0
        assert fr[b, x] > 0.0, (b, x)
        assert lo - CDF_TOL <= u <= cdf[x] + CDF_TOL, (b, x, xw, u, lo, cdf[x])
        lo_w = cdf[xw - 1] if xw > 0 else 0.0
        if lo_w + CDF_TOL < u < cdf[xw] - CDF_TOL:
            assert x == xw, (b, x, xw)
            exact += 1
    if V <= 1100:  # bins wide enough that most draws are strict comparisons
        assert exact >= max(1, int(clear.sum()) // 2), (exact, int(clear.sum()))
    return want_acc


def _uniforms(rng, total):
    return rng.random(total), rng.random(total)


@pytest.mark.parametrize("seed,nseq,N,W,V,budgets", [
    (1, 6, 4, 3, 500, (40, 1, 13, 40, 7, 30)),
    (2, 4, 6, 2, 1001, (60, 33, 2, 64)),
    (3, 3, 5, 4, 4099, (100, 256, 17)),
])
def test_matches_oracle_on_built_trees(seed, nseq, N, W, V, budgets):
    o = dict(nseq=nseq, N=N, W=W, V=V, budgets=budgets, prefix=("fixed", 0), Hq=4, Hkv=1, D=64,
             dtype="f32", qkv_std=1.0)
    wl = wk.make(1, seed=seed, overrides=o)
    tree = oracle_tree(wl)
    target = wk.target_logits(wl, tree["parent"], tree["token"])
    rng = np.random.default_rng(seed + 50)
    ua, ub = _uniforms(rng, wl.total)
    _compare(target, wl.draft_logits, tree["parent"], tree["token"], wl.tree_off, N, ua, ub)


def test_draft_rows_close_to_target_accept_deep_paths():
    """Target rows equal to the draft rows of the next depth (plus noise):
    acceptance probabilities are high and long paths are exercised."""
    rng = np.random.default_rng(9)
    o = dict(nseq=4, N=6, W=3, V=700, budgets=(120,), prefix=("fixed", 0), Hq=4, Hkv=1, D=64,
             dtype="f32", qkv_std=1.0)
    wl = wk.make(1, seed=9, overrides=o)
    tree = oracle_tree(wl)
    depth = np.zeros(wl.total, np.int64)
    for b in range(wl.nseq):
        off = wl.tree_off[b]
        for n in range(1, wl.tree_off[b + 1] - off):
            depth[off + n] = depth[off + tree["parent"][off + n]] + 1
    target = np.empty((wl.total, o["V"]), np.float32)
    for b in range(wl.nseq):
        for g in range(wl.tree_off[b], wl.tree_off[b + 1]):
            d = min(depth[g], o["N"] - 1)
            target[g] = wl.draft_logits[b, d] + rng.normal(0, 0.05, o["V"]).astype(np.float32)
    ua, ub = _uniforms(rng, wl.total)
    acc = _compare(target, wl.draft_logits, tree["parent"], tree["token"], wl.tree_off, o["N"], ua, ub)
    assert acc.max() >= 3


def test_full_vocabulary_verify_step():
    """Vocabulary 151936 (several vocabulary chunks per cluster CTA), eight
    trees of 256 nodes from the verify-step workload."""
    wl = wk.make(5)
    tree = oracle_tree(wl)
    target = wk.target_logits(wl, tree["parent"], tree["token"], deep=True)
    rng = np.random.default_rng(55)
    ua, ub = _uniforms(rng, wl.total)
    _compare(target, wl.draft_logits, tree["parent"], tree["token"], wl.tree_off, wl.cfg["N"], ua, ub)


def test_root_only_tree_draws_from_the_target_row():
    V = 64
    rng = np.random.default_rng(4)
    target = rng.normal(0, 1, (3, V)).astype(np.float32)
    draft = rng.normal(0, 1, (3, 2, V)).astype(np.float32)
    parent = np.array([-1, -1, -1], np.int32)
    token = np.array([5, 6, 7], np.int32)
    off = np.array([0, 1, 2, 3], np.int32)
    ua, ub = _uniforms(rng, 3)
    acc = _compare(target, draft, parent, token, off, 2, ua, ub)
    assert np.all(acc == 0)


def test_invalid_tree_is_flagged():
    z = torch.zeros((3, 8), dtype=torch.float32, device="cuda")
    d = torch.zeros((1, 2, 8), dtype=torch.float32, device="cuda")
    ws = jt.workspace(jt.jt_workspace_size(jt.JT_OP_VERIFY_ACCEPT, 1, 0, 0, 0, 3))
    u = torch.zeros(3, dtype=torch.float64, device="cuda")
    jt.jt_verify_accept_stochastic(z, d, dev(np.array([-1, 2, 0], np.int32)), dev(np.array([0, 1, 2], np.int32)),
                                   dev(np.array([0, 3], np.int32)), 2, u, u, ws=ws)
    with pytest.raises(jt.JtError):
        jt.jt_check(ws)
