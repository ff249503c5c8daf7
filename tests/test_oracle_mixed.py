"""Pins for the oracle's entropy-mixed tree build ("加速AI思考…" section 五
reports scoring by per-position entropy and by a weighted mix of cumulative
probability and entropy).  Reading: each step adds
(1 - alpha) * log-prob - alpha * H(draft row of the step's depth)."""
import itertools

import numpy as np
import pytest
from scipy.stats import entropy as scipy_entropy
from scipy.special import log_softmax

import oracle


def _draft(rng, nseq, N, V, scale=1.5):
    return (rng.standard_normal((nseq, N, V)) * scale).astype(np.float32)


def test_alpha_zero_is_the_plain_build():
    rng = np.random.default_rng(1)
    z = _draft(rng, 2, 4, 50)
    root = np.array([3, 4], np.int32)
    off = np.array([0, 20, 31], np.int32)
    a = oracle.tree_build(z, root, off, 3)
    b = oracle.tree_build_mixed(z, root, off, 3, 0.0)
    for k in ("parent", "token", "depth", "anc"):
        np.testing.assert_array_equal(a[k], b[k])


def test_entropy_matches_scipy():
    rng = np.random.default_rng(2)
    z = _draft(rng, 2, 3, 200)
    out = oracle.tree_build_mixed(z, np.zeros(2, np.int32), np.array([0, 5, 9], np.int32), 2, 0.3)
    p = np.exp(log_softmax(z.astype(np.float64), axis=-1))
    np.testing.assert_allclose(out["entropy"], scipy_entropy(p, axis=-1), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("alpha", [0.2, 0.5, 0.9, 1.0])
def test_matches_exhaustive_enumeration(alpha):
    """Nodes 1..B-1 are the B-1 best paths under the mixed step scores
    (sorted by score desc, depth asc, token asc, parent index asc), for
    every budget of small trees."""
    rng = np.random.default_rng(int(alpha * 10))
    for trial in range(12):
        N, W, V = int(rng.integers(1, 4)), int(rng.integers(1, 4)), int(rng.integers(5, 30))
        z = _draft(rng, 1, N, V, scale=float(rng.uniform(0.5, 3)))
        lp_full = log_softmax(z[0].astype(np.float64), axis=-1)
        H = scipy_entropy(np.exp(lp_full), axis=-1)
        order = np.lexsort((np.arange(V)[None, :].repeat(N, 0), -z[0]), axis=-1)[:, :W]
        full = sum(W ** d for d in range(N + 1))
        for B in range(1, full + 1):
            out = oracle.tree_build_mixed(z, np.array([7], np.int32), np.array([0, B], np.int32), W, alpha)
            # enumerate every path (k_1..k_d) with its score in root-to-node order
            paths = []
            for d in range(1, N + 1):
                for ks in itertools.product(range(W), repeat=d):
                    s = 0.0
                    for dd, k in enumerate(ks):
                        s = s + ((1.0 - alpha) * lp_full[dd, order[dd, k]] - alpha * H[dd])
                    paths.append((ks, s))
            # best-first pop order: the parent is placed first, so compare
            # by (score desc, depth asc, token asc, position of parent)
            placed = {(): 0}
            got = []
            remaining = list(paths)
            for n in range(1, B):
                cand = [(ks, s) for ks, s in remaining if ks[:-1] in placed]
                cand.sort(key=lambda t: (-t[1], len(t[0]), int(order[len(t[0]) - 1, t[0][-1]]),
                                         placed[t[0][:-1]]))
                ks, s = cand[0]
                placed[ks] = n
                got.append(ks)
                remaining.remove((ks, s))
            want_tok = [int(order[len(ks) - 1, ks[-1]]) for ks in got]
            want_par = [placed[ks[:-1]] for ks in got]
            np.testing.assert_array_equal(out["token"][1:], want_tok)
            np.testing.assert_array_equal(out["parent"][1:], want_par)


def test_alpha_outside_range_is_rejected():
    z = np.zeros((1, 1, 5), np.float32)
    for a in (-0.1, 1.0 + 1e-12, float("nan")):
        with pytest.raises(oracle.OracleError):
            oracle.tree_build_mixed(z, np.zeros(1, np.int32), np.array([0, 2], np.int32), 2, a)


def test_masked_entries_add_nothing_to_the_entropy():
    """Logits of -inf (probability 0) contribute 0 log 0 = 0: the entropy of
    a row with masked entries is that of its finite part, and a row with one
    finite entry has entropy 0."""
    rng = np.random.default_rng(5)
    z = _draft(rng, 1, 3, 120)
    z[0, 0, ::3] = -np.inf
    z[0, 1, :] = -np.inf
    z[0, 1, 17] = 4.0
    out = oracle.tree_build_mixed(z, np.zeros(1, np.int32), np.array([0, 4], np.int32), 1, 0.5)
    fin = z[0, 0][np.isfinite(z[0, 0])].astype(np.float64)
    np.testing.assert_allclose(out["entropy"][0, 0], scipy_entropy(np.exp(log_softmax(fin))), rtol=1e-12)
    assert out["entropy"][0, 1] == 0.0
    assert np.isfinite(out["entropy"]).all()


def test_pure_entropy_is_breadth_first_by_token():
    """alpha = 1: every node of depth d scores -(H_0 + ... + H_{d-1}) whatever
    its tokens, so with all H_d > 0 the queue's tie-breaks alone order a
    depth: the tree is breadth-first, a depth's nodes by (token asc, parent
    asc).  Closed form, independent of the entropy values."""
    rng = np.random.default_rng(11)
    N, W, V = 3, 3, 40
    z = _draft(rng, 1, N, V)
    order = np.lexsort((np.arange(V)[None, :].repeat(N, 0), -z[0]), axis=-1)[:, :W]
    full = 1 + W + W * W + W ** 3
    out = oracle.tree_build_mixed(z, np.array([5], np.int32), np.array([0, full], np.int32), W, 1.0)
    par, tok, dep = [0 - 1], [5], [0]
    level = [0]
    for d in range(N):
        kids = sorted(((int(t), p) for p in level for t in order[d]), key=lambda c: (c[0], c[1]))
        level = []
        for t, p in kids:
            level.append(len(tok))
            par.append(p)
            tok.append(t)
            dep.append(d + 1)
    np.testing.assert_array_equal(out["parent"], par)
    np.testing.assert_array_equal(out["token"], tok)
    np.testing.assert_array_equal(out["depth"], dep)


def test_zero_probability_candidates_come_last():
    """A row with fewer finite logits than W: the extra candidates have
    probability 0 and score -inf under every weight, so they are popped
    only once every finite path is in the tree."""
    V, W = 10, 4
    z = np.full((1, 2, V), -np.inf, np.float32)
    z[0, 0, [2, 6]] = [1.0, 0.5]
    z[0, 1, :] = np.linspace(0, 1, V, dtype=np.float32)
    for alpha in (0.0, 0.5, 1.0):
        out = oracle.tree_build_mixed(z, np.array([0], np.int32), np.array([0, 13], np.int32), W, alpha)
        # nodes 1..10: the two finite depth-1 nodes and their 8 children
        assert set(out["token"][1:3]) == {2, 6} and np.all(out["depth"][1:3] == 1)
        assert np.all(out["depth"][3:11] == 2) and np.all(np.isin(out["parent"][3:11], [1, 2]))
        assert np.all(out["score"][:11] > -np.inf) and np.all(out["score"][11:] == -np.inf)
