"""GPU parity of jt_verify_accept against the oracle: bit-exact accepted
length, path and bonus token, for the greedy rule and the margin rule
(AdaptiveSpec "逐步Margin规则")."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_jt_gb300 as jt
from tree_speculative_decoding_jt_gb300 import workloads as wk
from gpu_util import dev, oracle_tree

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _gpu(z, parent, token, off, N, rule, log_t):
    acc, path, bonus = jt.jt_verify_accept(dev(z), dev(parent), dev(token), dev(off), N, rule=rule,
                                           log_t=log_t)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), path.cpu().numpy(), bonus.cpu().numpy()


def _compare(z, parent, token, off, N, rule, log_t):
    got = _gpu(z, parent, token, off, N, rule, log_t)
    want = oracle.verify_accept(z, parent, token, off, N, rule, log_t)
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)
    return got


def test_margin_worked_example():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "margin_worked_example.txt"))
            if l.strip() and not l.startswith("#")]
    for p_top1, p_draft, t, _, accepted in rows:
        p = np.array([float(p_top1), float(p_draft)] + [0.05] * 7)
        z = np.log(p).astype(np.float32)[None].repeat(2, 0)
        acc, path, bonus = _compare(z, np.array([-1, 0], np.int32), np.array([5, 1], np.int32),
                                    np.array([0, 2], np.int32), 1, 1, math.log(float(t)))
        assert acc[0] == int(accepted)


def _random_batch(seed, nseq, V, deep):
    rng = np.random.default_rng(seed)
    parents, tokens, budgets = [], [], []
    for b in range(nseq):
        B = int(rng.integers(1, 257))
        par = np.full(B, -1, np.int32)
        tok = np.zeros(B, np.int32)
        tok[0] = rng.integers(0, V)
        used = {}
        for n in range(1, B):
            while True:
                p = int(rng.integers(max(0, n - 20), n))
                t = int(rng.integers(0, V))
                if t not in used.setdefault(p, set()):
                    break
            used[p].add(t)
            par[n], tok[n] = p, t
        parents.append(par)
        tokens.append(tok)
        budgets.append(B)
    off = np.concatenate([[0], np.cumsum(budgets)]).astype(np.int32)
    parent, token = np.concatenate(parents), np.concatenate(tokens)
    z = (rng.standard_normal((int(off[-1]), V)) * np.sqrt(2)).astype(np.float32)
    for b in range(nseq):
        for c in range(int(off[b]) + 1, int(off[b + 1])):
            if rng.random() < 0.8:
                row = int(off[b]) + int(parent[c])
                z[row, token[c]] = (z[row].max() + 0.05) if deep else z[row, token[c]] + 3.0
    depth = np.zeros(len(parent), np.int32)
    for b in range(nseq):
        o = int(off[b])
        for n in range(1, budgets[b]):
            depth[o + n] = depth[o + parent[o + n]] + 1
    return z, parent, token, off, int(depth.max())


@pytest.mark.parametrize("rule", [0, 1])
@pytest.mark.parametrize("deep", [False, True])
@pytest.mark.parametrize("V", [64, 4097])
def test_random_trees_match_oracle(rule, deep, V):
    z, parent, token, off, N = _random_batch(7 + V + rule + 2 * deep, 24, V, deep)
    for t in (0.8, 0.3, 1.0):
        _compare(z, parent, token, off, N, rule, math.log(t))


@pytest.mark.parametrize("cfg", [1, 2, 4, 5])
@pytest.mark.parametrize("deep", [False, True])
def test_config_trees_match_oracle(cfg, deep):
    """Full-size verify steps (config 4: 32 trees, 1.24 GB of target
    logits), greedy and margin, against the oracle on every sequence."""
    wl = wk.make(cfg, with_kv=False)
    tree = oracle_tree(wl)
    z = wk.target_logits(wl, tree["parent"], tree["token"], deep=deep)
    N = wl.cfg["N"]
    for rule in (0, 1):
        acc, _, _ = _compare(z, tree["parent"], tree["token"], wl.tree_off, N, rule,
                             math.log(wl.cfg["t"]))
        if deep:
            assert acc.max() >= 2


def test_invalid_tree_is_flagged():
    z = np.zeros((3, 8), np.float32)
    ws = jt.workspace(jt.jt_workspace_size(jt.JT_OP_VERIFY_ACCEPT, 1, 0, 0, 0, 3))
    jt.jt_verify_accept(dev(z), dev(np.array([-1, 2, 0], np.int32)), dev(np.array([0, 1, 2], np.int32)),
                        dev(np.array([0, 3], np.int32)), 2, ws=ws)
    with pytest.raises(jt.JtError):
        jt.jt_check(ws)


def test_deepest_paths_at_maximum_depth():
    """Chains of 64 drafted nodes whose target rows all pick the drafted
    token: both rules accept the whole chain (accept_len 64, path of 65)."""
    N, V, nseq = 64, 300, 3
    rng = np.random.default_rng(64)
    token = rng.integers(0, V, size=(nseq, N + 1)).astype(np.int32).reshape(-1)
    parent = np.tile(np.arange(-1, N, dtype=np.int32), nseq)
    off = (np.arange(nseq + 1) * (N + 1)).astype(np.int32)
    z = rng.standard_normal((nseq * (N + 1), V)).astype(np.float32)
    for b in range(nseq):
        for c in range(1, N + 1):
            row = off[b] + c - 1
            z[row, token[off[b] + c]] = z[row].max() + 2.0
    for rule in (0, 1):
        acc, path, _ = _compare(z, parent, token, off, N, rule, math.log(0.8))
        assert np.all(acc == N)
        np.testing.assert_array_equal(path[:, -1], N)
