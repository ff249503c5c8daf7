"""Pins for the oracle's capped expansion and adaptive tree policy
("AdaptiveSpec：免训练推测解码方案提速56%的技术解析", section on the per-step
tree policy: the draft's top-1 confidence and the rolling acceptance history
set depth, width and node count; the tree grows when both are high and
shrinks in the opposite case.  "加速AI思考…" section 七: large budgets stop
paying as the batch grows).

The caps are pinned by a different route (the plain expansion of truncated
tables); the policy by closed forms (the EMA, doubling and halving runs),
by the page's direction (the emitted budget never falls when a signal
rises) and by its invariants (feasible budgets, prefix sums, the load cap)."""
import numpy as np
import pytest

import oracle

P = oracle.POLICY_DEFAULTS


def _tables(rng, nseq, N, W):
    lp = -np.sort(rng.exponential(1.0, size=(nseq, N, W)), axis=2)
    tok = np.stack([np.stack([rng.choice(5000, size=W, replace=False) for _ in range(N)])
                    for _ in range(nseq)]).astype(np.int32)
    return tok, lp


def _full(n, w):
    return sum(w ** d for d in range(n + 1))


# ---------------------------------------------------------------- caps


def test_caps_at_the_table_size_change_nothing():
    rng = np.random.default_rng(1)
    tok, lp = _tables(rng, 3, 5, 3)
    root = np.array([1, 2, 3], np.int32)
    off = np.array([0, 40, 41, 160], np.int32)
    a = oracle.tree_expand(tok, lp, root, off, 5, 3)
    b = oracle.tree_expand_capped(tok, lp, root, off, 5, 3, w_cap=[3, 3, 3], n_cap=[5, 5, 5])
    for k in ("parent", "token", "depth", "anc", "score"):
        np.testing.assert_array_equal(a[k], b[k])


@pytest.mark.parametrize("seed", range(8))
def test_caps_equal_the_plain_expansion_of_truncated_tables(seed):
    """Sequence b under caps (w, n) is the plain expansion of its table cut
    to the first n rows and the first w candidates of each."""
    rng = np.random.default_rng(10 + seed)
    nseq, N, W = 4, 6, 4
    tok, lp = _tables(rng, nseq, N, W)
    if seed % 2:
        lp = np.round(lp, 1)             # ties decided by the queue key
    wc = rng.integers(1, W + 1, size=nseq).astype(np.int32)
    nc = rng.integers(0, N + 1, size=nseq).astype(np.int32)
    budgets = [int(rng.integers(1, min(_full(int(n), int(w)), 256) + 1)) for n, w in zip(nc, wc)]
    off = np.concatenate([[0], np.cumsum(budgets)]).astype(np.int32)
    root = rng.integers(0, 5000, size=nseq).astype(np.int32)
    got = oracle.tree_expand_capped(tok, lp, root, off, N, W, w_cap=wc, n_cap=nc)
    for b in range(nseq):
        n, w = int(nc[b]), int(wc[b])
        t = tok[b:b + 1, :n, :w] if n > 0 else np.zeros((1, 0, w), np.int32)
        l = lp[b:b + 1, :n, :w] if n > 0 else np.zeros((1, 0, w))
        want = oracle.tree_expand(t, l, root[b:b + 1], np.array([0, budgets[b]], np.int32), n, w)
        s = slice(off[b], off[b + 1])
        for k in ("parent", "token", "depth", "anc", "score"):
            np.testing.assert_array_equal(got[k][s], want[k], err_msg=f"{k} b={b}")


def test_caps_reject_budgets_beyond_the_capped_tree():
    rng = np.random.default_rng(2)
    tok, lp = _tables(rng, 1, 4, 3)
    root = np.array([0], np.int32)
    with pytest.raises(oracle.OracleError):       # full(2, 2) = 7
        oracle.tree_expand_capped(tok, lp, root, np.array([0, 8], np.int32), 4, 3, w_cap=[2], n_cap=[2])
    out = oracle.tree_expand_capped(tok, lp, root, np.array([0, 7], np.int32), 4, 3, w_cap=[2], n_cap=[2])
    assert out["depth"].max() == 2
    with pytest.raises(oracle.OracleError):
        oracle.tree_expand_capped(tok, lp, root, np.array([0, 2], np.int32), 4, 3, w_cap=[1], n_cap=[0])
    root_only = oracle.tree_expand_capped(tok, lp, root, np.array([0, 1], np.int32), 4, 3, n_cap=[0])
    assert list(root_only["parent"]) == [-1]
    for bad in ({"w_cap": [0]}, {"w_cap": [4]}, {"n_cap": [5]}, {"n_cap": [-1]}):
        with pytest.raises(oracle.OracleError):
            oracle.tree_expand_capped(tok, lp, root, np.array([0, 1], np.int32), 4, 3, **bad)


# ---------------------------------------------------------------- policy


def _lp_with_top1(p_top1, N=4, W=3):
    """Tables whose depth-1 top-1 log-probability is log(p_top1)."""
    p_top1 = np.asarray(p_top1, np.float64)
    lp = np.full((len(p_top1), N, W), -3.0)
    lp[:, 0, 0] = np.log(p_top1)
    return lp


def test_ema_closed_form():
    """A constant accepted length a: ema_t = a + (1 - beta)^t (ema_0 - a)."""
    lp = _lp_with_top1([0.9, 0.1])
    bs, ema = np.array([32, 32]), np.array([0.0, 4.0])
    acc = np.array([3, 1], np.int32)
    beta = 0.3
    for t in range(1, 25):
        r = oracle.tree_policy(lp, acc, bs, ema, beta=beta)
        bs, ema = r["budget_state"], r["acc_ema"]
        want = acc + (1 - beta) ** t * (np.array([0.0, 4.0]) - acc)
        np.testing.assert_allclose(ema, want, rtol=1e-12, atol=1e-12)


def test_unobserved_steps_leave_the_ema():
    lp = _lp_with_top1([0.9, 0.9])
    r = oracle.tree_policy(lp, np.array([-1, -1]), [16, 16], [2.5, 0.0])
    np.testing.assert_array_equal(r["acc_ema"], [2.5, 0.0])
    r2 = oracle.tree_policy(lp, None, [16, 16], [2.5, 0.0])
    np.testing.assert_array_equal(r2["acc_ema"], [2.5, 0.0])


def test_budget_doubles_halves_and_holds():
    """Confident and accepting: B_t = min(b_max, B_0 2^t); neither: B_t =
    max(b_min, floor(B_0 / 2^t)); signals that disagree: B unchanged."""
    N = 4
    lp = _lp_with_top1([0.9, 0.1, 0.9, 0.1], N=N)
    acc = np.array([N, 0, 0, N], np.int32)
    ema = np.array([float(N), 0.0, 0.0, float(N)])
    bs0 = np.array([20, 200, 50, 50], np.int32)
    bs = bs0.copy()
    for t in range(1, 8):
        r = oracle.tree_policy(lp, acc, bs, ema, b_min=16, b_max=256, beta=1.0)
        bs, ema = r["budget_state"], r["acc_ema"]
        assert bs[0] == min(256, 20 * 2 ** t)
        assert bs[1] == max(16, 200 // 2 ** t)
        assert bs[2] == 50 and bs[3] == 50


def test_state_is_clamped_into_the_bounds_first():
    lp = _lp_with_top1([0.9, 0.1])
    r = oracle.tree_policy(lp, None, [1000, 1], [3.0, 3.0], b_min=16, b_max=128)
    # conf & hot: clamp 1000 -> 128, double -> 128; not conf, hot: clamp 1 -> 16, hold
    np.testing.assert_array_equal(r["budget_state"], [128, 16])


def test_caps_follow_the_signals():
    N, W = 8, 4
    lp = _lp_with_top1([0.9, 0.2, 0.9, 0.9], N=N, W=W)
    ema = np.array([0.0, 0.0, 2.7, 30.0])
    r = oracle.tree_policy(lp, None, [64] * 4, ema, w_min=2, n_min=2, n_slack=3)
    np.testing.assert_array_equal(r["w_cap"], [W, 2, W, W])
    np.testing.assert_array_equal(r["n_cap"], [3, 3, 5, N])
    r = oracle.tree_policy(lp, None, [64] * 4, ema, w_min=2, n_min=4, n_slack=0)
    np.testing.assert_array_equal(r["n_cap"], [4, 4, 4, N])


@pytest.mark.parametrize("seed", range(6))
def test_invariants_and_load_cap(seed):
    rng = np.random.default_rng(seed)
    nseq, N, W = int(rng.integers(1, 40)), int(rng.integers(1, 10)), int(rng.integers(1, 6))
    lp = -np.sort(rng.exponential(0.7, size=(nseq, N, W)), axis=2)
    prm = dict(b_min=int(rng.integers(1, 20)), w_min=int(rng.integers(1, W + 1)),
               n_min=int(rng.integers(0, N + 1)), n_slack=int(rng.integers(0, N + 1)),
               beta=float(rng.uniform(0.05, 1.0)), log_conf=float(np.log(rng.uniform(0.2, 0.9))),
               acc_thresh=float(rng.uniform(0, N)), node_cap=int(rng.integers(0, 3000)))
    prm["b_max"] = int(rng.integers(prm["b_min"], 257))
    bs = rng.integers(1, 300, size=nseq)
    ema = rng.uniform(0, N, size=nseq)
    for _ in range(5):
        acc = rng.integers(-1, N + 1, size=nseq).astype(np.int32)
        r = oracle.tree_policy(lp, acc, bs, ema, **prm)
        off, wc, nc = r["tree_off"], r["w_cap"], r["n_cap"]
        emit = np.diff(off)
        assert off[0] == 0 and np.all(emit >= 1)
        assert np.all(emit <= [min(256, _full(int(n), int(w))) for n, w in zip(nc, wc)])
        assert np.all(emit <= r["budget_state"])
        ceil_b = prm["b_max"] if prm["node_cap"] == 0 else \
            min(prm["b_max"], max(prm["b_min"], prm["node_cap"] // nseq))
        assert np.all((r["budget_state"] >= prm["b_min"]) & (r["budget_state"] <= ceil_b))
        if prm["node_cap"] > 0:
            assert off[-1] <= max(prm["node_cap"], nseq * prm["b_min"])
        assert np.all((wc == W) | (wc == prm["w_min"]))
        assert np.all((nc >= prm["n_min"]) & (nc <= N))
        bs, ema = r["budget_state"], r["acc_ema"]


@pytest.mark.parametrize("seed", range(4))
def test_emitted_budget_never_falls_when_a_signal_rises(seed):
    """The page's direction: more confidence or more acceptance never gives
    a smaller tree (same state, one signal raised)."""
    rng = np.random.default_rng(50 + seed)
    nseq, N, W = 200, 6, 4
    lp = -np.sort(rng.exponential(0.7, size=(nseq, N, W)), axis=2)
    bs = rng.integers(1, 300, size=nseq)
    ema = rng.uniform(0, N, size=nseq)
    acc = rng.integers(0, N + 1, size=nseq).astype(np.int32)
    prm = dict(b_min=8, b_max=200, w_min=1, n_min=1, n_slack=2, acc_thresh=2.5, beta=0.5)
    base = np.diff(oracle.tree_policy(lp, acc, bs, ema, **prm)["tree_off"])
    lp_up = lp.copy()
    lp_up[:, 0, 0] = np.minimum(0.0, lp[:, 0, 0] + rng.uniform(0, 2, size=nseq))
    up_c = np.diff(oracle.tree_policy(lp_up, acc, bs, ema, **prm)["tree_off"])
    acc_up = np.minimum(N, acc + rng.integers(0, 3, size=nseq)).astype(np.int32)
    up_a = np.diff(oracle.tree_policy(lp, acc_up, bs, ema, **prm)["tree_off"])
    assert np.all(up_c >= base) and np.all(up_a >= base)
    assert np.any(up_c > base) and np.any(up_a > base)


def test_policy_feeds_the_capped_expansion():
    """Several steps of policy -> capped expansion: every tree respects its
    caps (depth <= n_cap, each token among the first w_cap of its row)."""
    rng = np.random.default_rng(77)
    nseq, N, W = 6, 8, 4
    bs, ema = np.full(nseq, 32), np.full(nseq, 2.0)
    acc = None
    for _ in range(6):
        tok, lp = _tables(rng, nseq, N, W)
        r = oracle.tree_policy(lp, acc, bs, ema, b_min=4, b_max=256, w_min=2, n_min=1, n_slack=2,
                               log_conf=float(np.log(0.6)), acc_thresh=2.0)
        off, wc, nc = r["tree_off"], r["w_cap"], r["n_cap"]
        root = rng.integers(0, 5000, size=nseq).astype(np.int32)
        t = oracle.tree_expand_capped(tok, lp, root, off, N, W, w_cap=wc, n_cap=nc)
        for b in range(nseq):
            s = slice(off[b] + 1, off[b + 1])
            assert np.all(t["depth"][s] <= nc[b])
            for tk, d in zip(t["token"][s], t["depth"][s]):
                assert tk in tok[b, d - 1, :wc[b]]
        acc = rng.integers(0, N + 1, size=nseq).astype(np.int32)
        bs, ema = r["budget_state"], r["acc_ema"]


def test_invalid_arguments_are_rejected():
    lp = _lp_with_top1([0.9])
    for bad in (dict(b_min=0), dict(b_max=257), dict(b_min=20, b_max=10), dict(w_min=4), dict(w_min=0),
                dict(n_min=5), dict(n_slack=5), dict(beta=0.0), dict(beta=1.5), dict(node_cap=-1),
                dict(log_conf=float("nan")), dict(acc_thresh=float("nan"))):
        with pytest.raises(oracle.OracleError):
            oracle.tree_policy(lp, None, [16], [1.0], **bad)
    for acc, ema in (([5], [1.0]), ([-2], [1.0]), ([1], [-0.5]), ([1], [float("nan")]),
                     ([1], [float("inf")])):
        with pytest.raises(oracle.OracleError):
            oracle.tree_policy(lp, acc, [16], ema)
