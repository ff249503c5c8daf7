"""Pins for the oracle's tree build (CPU only).

The oracle's top-W/lse is checked against numpy's sort and scipy's
logsumexp; its best-first expansion against exhaustive enumeration of every
path of the full tree (north star: "best-first expansion must match
exhaustive enumeration of paths for small B"), plus closed special cases.
"""
import itertools

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle


def test_topw_lse_matches_library_routines():
    rng = np.random.default_rng(1)
    for V, W in [(7, 1), (50, 3), (1000, 8), (4099, 4)]:
        z = (rng.standard_normal((6, V)) * 1.4).astype(np.float32)
        # plant ties so that the id tie-break matters
        z[0, 3] = z[0, 5] = z[0].max() + 1
        z[1, :] = 0.25
        tok, lp, lse = oracle.topw_lse(z, W)
        for r in range(z.shape[0]):
            order = np.lexsort((np.arange(V), -z[r].astype(np.float64)))  # value desc, id asc
            np.testing.assert_array_equal(tok[r], order[:W])
            ref = logsumexp(z[r].astype(np.float64))
            assert abs(lse[r] - ref) <= 1e-12 * max(1.0, abs(ref))
            np.testing.assert_allclose(lp[r], z[r, order[:W]].astype(np.float64) - ref,
                                       rtol=0, atol=1e-12)


def test_topw_lse_with_minus_inf_entries():
    z = np.full((1, 10), -np.inf, np.float32)
    z[0, 4] = 1.0
    z[0, 7] = 1.0
    tok, lp, lse = oracle.topw_lse(z, 3)
    assert list(tok[0, :2]) == [4, 7]
    assert abs(lse[0] - (1.0 + np.log(2.0))) < 1e-15
    assert lp[0, 2] == -np.inf


def _brute_force(tok, lp, N, W, B):
    """Every path of the full W-ary depth-N tree, scored by the same
    sequential fp64 sum root->leaf, sorted by (score desc, depth asc,
    token asc, then the parent's own key); returns the first B-1 paths as
    tuples of child ranks.  Ordering ties by the parent's key is ordering by
    parent index, because parents leave the queue in key order."""
    score = {}
    for d in range(1, N + 1):
        for ks in itertools.product(range(W), repeat=d):
            s = 0.0
            for depth, k in enumerate(ks):
                s = s + float(lp[depth, k])
            score[ks] = s

    def key(ks):
        parts, cur = [], ks
        while cur:
            parts.append((-score[cur], len(cur), int(tok[len(cur) - 1, cur[-1]])))
            cur = cur[:-1]
        return parts

    return sorted(score, key=key)[:B - 1]


@pytest.mark.parametrize("W", [1, 2, 3])
def test_expand_equals_exhaustive_enumeration(W):
    rng = np.random.default_rng(100 + W)
    for trial in range(200 if W > 1 else 40):
        N = int(rng.integers(1, 6))
        full = sum(W ** d for d in range(0, N + 1))
        if full > 256:
            N = max(1, N - 1)
            full = sum(W ** d for d in range(0, N + 1))
        B = int(rng.integers(1, min(full, 256) + 1))
        # per-depth tables: ids distinct per row, lp sorted desc (ties on
        # purpose in some trials)
        lp = -np.sort(rng.exponential(1.0, size=(N, W)), axis=1)
        if trial % 5 == 0:
            lp = np.round(lp, 1)
        tok = np.stack([np.sort(rng.choice(50, size=W, replace=False)) for _ in range(N)]).astype(np.int32)
        res = oracle.tree_expand(tok[None], lp[None], np.array([7]), np.array([0, B]), N, W)
        want = _brute_force(tok, lp, N, W, B)
        # the oracle's nodes as child-rank tuples (rank k of the child's token at its depth)
        got = []
        rank_of = [{int(t): k for k, t in enumerate(tok[d])} for d in range(N)]
        for n in range(1, B):
            ks, u = [], n
            while res["parent"][u] >= 0:
                ks.append(rank_of[res["depth"][u] - 1][int(res["token"][u])])
                u = res["parent"][u]
            got.append(tuple(reversed(ks)))
        assert got == want, (trial, N, W, B)
        assert res["parent"][0] == -1 and res["token"][0] == 7 and res["depth"][0] == 0


def test_expand_tiny_hand_worked():
    # depth-1 candidates: a (id 10, lp -0.1), b (id 11, lp -2.0);
    # depth-2 candidates: x (id 20, lp -0.5), y (id 21, lp -0.7).
    # paths: a=-0.1, a.x=-0.6, a.y=-0.8, b=-2.0, b.x=-2.5, b.y=-2.7
    tok = np.array([[[10, 11], [20, 21]]], np.int32)
    lp = np.array([[[-0.1, -2.0], [-0.5, -0.7]]])
    res = oracle.tree_expand(tok, lp, np.array([1]), np.array([0, 5]), 2, 2)
    assert list(res["parent"]) == [-1, 0, 1, 1, 0]
    assert list(res["token"]) == [1, 10, 20, 21, 11]
    assert list(res["depth"]) == [0, 1, 2, 2, 1]
    np.testing.assert_allclose(res["score"], [0.0, -0.1, -0.6, -0.8, -2.0], atol=1e-15)
    # ancestor-or-self sets
    assert list(res["anc"][:, 0]) == [0b1, 0b11, 0b111, 0b1011, 0b10001]


def test_w1_chain_and_b1_root_only():
    rng = np.random.default_rng(5)
    z = rng.standard_normal((1, 6, 300)).astype(np.float32) * 1.4
    res = oracle.tree_build(z, np.array([3]), np.array([0, 5]), 1)
    assert list(res["parent"]) == [-1, 0, 1, 2, 3]
    assert list(res["token"][1:]) == [int(np.argmax(z[0, d])) for d in range(4)]
    res1 = oracle.tree_build(z, np.array([3]), np.array([0, 1]), 4)
    assert list(res1["parent"]) == [-1] and list(res1["token"]) == [3]


def test_budget_beyond_full_tree_is_rejected():
    z = np.zeros((1, 2, 10), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.tree_build(z, np.array([0]), np.array([0, 8]), 2)  # full tree has 7 nodes
    res = oracle.tree_build(z, np.array([0]), np.array([0, 7]), 2)
    assert sorted(res["depth"]) == [0, 1, 1, 2, 2, 2, 2]


def test_invariants_on_config_shaped_trees():
    rng = np.random.default_rng(9)
    nseq, N, W, V = 3, 16, 4, 2000
    z = (rng.standard_normal((nseq, N, V)) * np.sqrt(2)).astype(np.float32)
    budgets = [256, 100, 37]
    off = np.concatenate([[0], np.cumsum(budgets)]).astype(np.int32)
    res = oracle.tree_build(z, np.array([1, 2, 3]), off, W)
    for b in range(nseq):
        o, B = off[b], budgets[b]
        par, dep, sc = res["parent"][o:o + B], res["depth"][o:o + B], res["score"][o:o + B]
        assert par[0] == -1
        for n in range(1, B):
            assert 0 <= par[n] < n
            assert dep[n] == dep[par[n]] + 1 <= N
        assert np.all(np.diff(sc) <= 0), "pop order must be non-increasing in score"
        for n in range(B):
            sib = [c for c in range(B) if par[c] == par[n]]
            assert len({int(res["token"][o + c]) for c in sib}) == len(sib)
        assert res["gap"][b] >= 0
