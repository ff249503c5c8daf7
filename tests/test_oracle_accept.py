"""Pins for the oracle's tree acceptance (CPU only).

Greedy rule ("加速AI思考…" section 三; JetSpec summary): along each path keep
the longest prefix the target agrees with, adopt the longest.  Margin rule
(AdaptiveSpec, section "逐步Margin规则"): accept a drafted token when
p_target(draft)/p_target(top1) >= t.  Checked against the pages' worked
example and closed form, and against brute-force enumeration of paths with
numpy's argmax.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(path):
    out = []
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            out.append([float(x) for x in line.split()])
    return out


def test_margin_worked_example():
    for p_top1, p_draft, t, ratio, accepted in _rows(os.path.join(GOLDEN, "margin_worked_example.txt")):
        assert round(p_draft / p_top1, 2) == ratio
        # row of the root: token 0 is top-1 (0.35), token 1 the draft (0.30),
        # the remaining 0.35 spread over 7 tokens of 0.05
        p = np.array([p_top1, p_draft] + [0.05] * 7)
        z = np.log(p).astype(np.float32)[None].repeat(2, 0)
        parent = np.array([-1, 0], np.int32)
        token = np.array([5, 1], np.int32)
        acc, path, bonus = oracle.verify_accept(z, parent, token, np.array([0, 2]), 1, 1, np.log(t))
        assert acc[0] == int(accepted)
        assert list(path[0]) == ([0, 1] if accepted else [0, -1])
        assert bonus[0] == 0
        # the greedy rule rejects it: the draft is not the argmax
        acc_g, _, _ = oracle.verify_accept(z, parent, token, np.array([0, 2]), 1, 0)
        assert acc_g[0] == 0


def test_chain_acceptance_length_closed_form():
    """A W=1 chain of length 16 where each drafted token is the target's
    argmax with probability 0.85: P(all 16 accepted) = 0.85**16 ~ 0.074
    (the page rounds it to about 8%), and P(len = k) = 0.85**k * 0.15."""
    (p_match, n, approx), = _rows(os.path.join(GOLDEN, "chain_acceptance_closed_form.txt"))
    n = int(n)
    assert abs(p_match ** n - approx) < 0.01
    rng = np.random.default_rng(21)
    trials, V = 3000, 6
    nodes = n + 1
    parent = np.tile(np.arange(-1, n, dtype=np.int32), trials)
    token = np.tile(np.full(nodes, 2, np.int32), trials)
    off = np.arange(trials + 1, dtype=np.int32) * nodes
    z = rng.standard_normal((trials * nodes, V)).astype(np.float32)
    match = rng.random(trials * nodes) < p_match
    z[:, 2] = np.where(match, z.max(axis=1) + 1.0, z.min(axis=1) - 1.0)
    acc, _, _ = oracle.verify_accept(z, parent, token, off, n, 0)
    hist = np.bincount(acc, minlength=n + 1) / trials
    expect = np.array([p_match ** k * (1 - p_match) for k in range(n)] + [p_match ** n])
    sd = np.sqrt(expect * (1 - expect) / trials)
    assert np.all(np.abs(hist - expect) <= 4.5 * sd + 1e-9), (hist, expect)


def _random_tree(rng, B, V):
    parent = np.full(B, -1, np.int32)
    token = np.zeros(B, np.int32)
    token[0] = rng.integers(0, V)
    for n in range(1, B):
        for _ in range(100):
            p = int(rng.integers(0, n))
            used = {int(token[c]) for c in range(1, n) if parent[c] == p}
            free = [t for t in range(V) if t not in used]
            if free:
                break
        parent[n] = p
        token[n] = rng.choice(free)
    return parent, token


def _brute(z, parent, token, rule, log_t):
    """Enumerate every root->node path; a path is accepted when each edge
    passes the rule at its parent's row; return the deepest accepted node
    (lowest index on ties)."""
    B = len(parent)
    best, best_depth = 0, 0
    for n in range(B):
        path = []
        u = n
        while u >= 0:
            path.append(u)
            u = parent[u]
        path = path[::-1]
        ok = True
        for a, c in zip(path[:-1], path[1:]):
            row = z[a].astype(np.float64)
            if rule == 0:
                ok &= int(np.argmax(z[a])) == int(token[c])
            else:
                ok &= (row[token[c]] - row.max()) >= log_t
        if ok and len(path) - 1 > best_depth:
            best, best_depth = n, len(path) - 1
    return best, best_depth


@pytest.mark.parametrize("rule", [0, 1])
def test_accept_equals_brute_force(rule):
    rng = np.random.default_rng(30 + rule)
    for trial in range(300):
        B = int(rng.integers(1, 40))
        V = int(rng.integers(3, 12))
        parent, token = _random_tree(rng, B, V)
        z = rng.standard_normal((B, V)).astype(np.float32)
        if trial % 3 == 0:  # make many edges pass: boost drafted tokens to near the max
            for c in range(1, B):
                if rng.random() < 0.8:
                    z[parent[c], token[c]] = z[parent[c]].max() + (0.5 if rule == 0 else -0.1)
        if trial % 7 == 0:  # ties in the row maximum (argmax ties go to the lowest id)
            z[:, :2] = z.max(axis=1, keepdims=True)
        log_t = float(np.log(rng.uniform(0.3, 1.0)))
        depth = np.zeros(B, np.int32)
        for n in range(1, B):
            depth[n] = depth[parent[n]] + 1
        N = int(depth.max())
        acc, path, bonus = oracle.verify_accept(z, parent, token, np.array([0, B]), N, rule, log_t)
        fin, d = _brute(z, parent, token, rule, log_t)
        assert acc[0] == d, trial
        if rule == 1:
            assert path[0, d] == fin
        # the path is the root->final chain, padded with -1
        chain = []
        u = path[0, d]
        while u >= 0:
            chain.append(u)
            u = parent[u]
        assert list(path[0, :d + 1]) == chain[::-1] and all(path[0, d + 1:] == -1)
        assert bonus[0] == int(np.argmax(z[path[0, d]]))


def test_margin_at_t1_equals_greedy_without_ties():
    rng = np.random.default_rng(40)
    for trial in range(100):
        B, V = int(rng.integers(2, 60)), 9
        parent, token = _random_tree(rng, B, V)
        z = rng.standard_normal((B, V)).astype(np.float32)
        for c in range(1, B):
            if rng.random() < 0.7:
                z[parent[c], token[c]] = z[parent[c]].max() + 1.0
        depth = np.zeros(B, np.int32)
        for n in range(1, B):
            depth[n] = depth[parent[n]] + 1
        N = int(depth.max())
        g = oracle.verify_accept(z, parent, token, np.array([0, B]), N, 0)
        m = oracle.verify_accept(z, parent, token, np.array([0, B]), N, 1, 0.0)
        for a, b in zip(g, m):
            assert np.array_equal(a, b), trial


def test_non_topological_tree_is_rejected():
    z = np.zeros((3, 4), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.verify_accept(z, np.array([-1, 2, 0]), np.array([0, 1, 2]), np.array([0, 3]), 2, 0)
