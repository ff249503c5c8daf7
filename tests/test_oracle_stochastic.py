"""Pins for the oracle's temperature-1 tree acceptance (rejection sampling
against a running residual; the speculative-decoding overview's acceptance
section and AdaptiveSpec's section on the strict verification rule).

The strongest pin is the property the rule exists for: when the candidate
tokens are drawn i.i.d. from the draft distribution q, the first emitted
token (the accepted child's token, else the bonus drawn from the residual)
is distributed exactly as the target p.  A wrong residual, a missing
renormalisation or a wrong inverse CDF breaks it."""
import numpy as np
import pytest

import oracle


def _softmax(z):
    e = np.exp(z - z.max())
    return e / e.sum()


def _chain_batch(p, q, k, trials, rng, p_child=None):
    """`trials` one-level trees: a root with k children whose tokens are
    i.i.d. draws from q (N = 1, so children are leaves)."""
    V = len(p)
    B = 1 + k
    nseq = trials
    zt = np.log(np.maximum(p, 1e-300)).astype(np.float32)
    zc = np.log(np.maximum(p_child if p_child is not None else np.full(V, 1.0 / V), 1e-300)).astype(np.float32)
    target = np.empty((nseq * B, V), np.float32)
    target[:] = zc
    target[::B] = zt
    draft = np.broadcast_to(np.log(q).astype(np.float32), (nseq, 1, V)).copy()
    parent = np.tile(np.array([-1] + [0] * k, np.int32), nseq)
    tok = rng.choice(V, size=(nseq, k), p=q).astype(np.int32)
    token = np.concatenate([np.zeros((nseq, 1), np.int32), tok], axis=1).reshape(-1)
    off = (np.arange(nseq + 1) * B).astype(np.int32)
    ua = rng.random(nseq * B)
    ub = rng.random(nseq * B)
    return target, draft, parent, token, off, ua, ub


def _first_tokens(acc, path, bonus, token, off):
    first = bonus.copy()
    hit = acc >= 1
    first[hit] = token[off[:-1][hit] + path[hit, 1]]
    return first


@pytest.mark.parametrize("k", [1, 2, 4])
def test_first_token_is_distributed_as_the_target(k):
    rng = np.random.default_rng(100 + k)
    V, trials = 6, 60000
    p = _softmax(rng.normal(0, 1.2, V))
    q = _softmax(rng.normal(0, 1.2, V))
    target, draft, parent, token, off, ua, ub = _chain_batch(p, q, k, trials, rng)
    acc, path, bonus, _ = oracle.verify_accept_stochastic(target, draft, parent, token, off, 1, ua, ub)
    first = _first_tokens(acc, path, bonus, token, off)
    freq = np.bincount(first, minlength=V) / trials
    sigma = np.sqrt(p * (1 - p) / trials)
    assert np.all(np.abs(freq - p) <= 5 * sigma + 1e-4), (freq, p)
    # acceptance of the first child alone: probability sum_x min(p, q)
    first_child_taken = (acc >= 1) & (path[:, 1] == 1)
    want = np.minimum(p, q).sum()
    assert abs(first_child_taken.mean() - want) <= 5 * np.sqrt(want * (1 - want) / trials)


def test_second_token_follows_the_accepted_childs_row():
    """q = p at the root: the first child is always accepted; the bonus is
    then drawn from the child's own target row."""
    rng = np.random.default_rng(7)
    V, trials = 5, 40000
    p = _softmax(rng.normal(0, 1, V))
    pc = _softmax(rng.normal(0, 1, V))
    target, draft, parent, token, off, ua, ub = _chain_batch(p, p, 1, trials, rng, p_child=pc)
    acc, path, bonus, _ = oracle.verify_accept_stochastic(target, draft, parent, token, off, 1, ua, ub)
    assert np.all(acc == 1)
    freq = np.bincount(bonus, minlength=V) / trials
    assert np.all(np.abs(freq - pc) <= 5 * np.sqrt(pc * (1 - pc) / trials) + 1e-4)


def test_hand_worked_residual():
    """p = (.5, .5, 0), q = (.2, .3, .5); the child drafts token 2, which p
    rules out: rejected whatever u is; residual = (.3, .2, 0) / .5 =
    (.6, .4, 0), so u_bonus = .55 gives token 0 and .65 gives token 1."""
    p = np.array([0.0, 0.0, -200.0], np.float32)       # softmax (.5, .5, ~7e-88)
    q = np.log(np.array([[[0.2, 0.3, 0.5]]], np.float32))
    target = np.stack([p, np.zeros(3, np.float32)])
    for ub, want in ((0.55, 0), (0.65, 1), (0.05, 0), (0.95, 1)):
        acc, path, bonus, margin = oracle.verify_accept_stochastic(
            target, q, np.array([-1, 0]), np.array([0, 2]), np.array([0, 2]), 1,
            np.array([0.0, 0.5]), np.array([ub, 0.0]))
        assert acc[0] == 0 and path[0, 0] == 0 and path[0, 1] == -1
        assert bonus[0] == want
        assert margin[0] == pytest.approx(0.5)   # |u_accept - min(1, ratio ~ 1e-87)|
    _, _, _, _, fr, fu = oracle.verify_accept_stochastic(
        target, q, np.array([-1, 0]), np.array([0, 2]), np.array([0, 2]), 1,
        np.array([0.0, 0.5]), np.array([0.3, 0.0]), with_residual=True)
    np.testing.assert_allclose(fr[0], [0.6, 0.4, 0.0], atol=1e-7)
    assert fu[0] == 0.3


def test_draft_equal_to_target_always_accepts_and_leaf_samples_its_row():
    rng = np.random.default_rng(3)
    V = 7
    z = rng.normal(0, 1, V).astype(np.float32)
    # chain of depth 3 whose draft rows equal the target rows of the parents
    target = np.stack([z, z, z, z])
    draft = np.stack([z, z, z])[None]
    parent = np.array([-1, 0, 1, 2], np.int32)
    token = np.array([0, 3, 1, 6], np.int32)
    for _ in range(20):
        ua, ub = rng.random(4) * 0.999, rng.random(4)
        acc, path, bonus, _ = oracle.verify_accept_stochastic(target, draft, parent, token,
                                                              np.array([0, 4]), 3, ua, ub)
        assert acc[0] == 3 and list(path[0]) == [0, 1, 2, 3]
        cdf = np.cumsum(_softmax(z.astype(np.float64)))
        assert bonus[0] == int(np.searchsorted(cdf, ub[3] * cdf[-1], side="right"))


def test_invalid_trees_are_rejected():
    z = np.zeros((2, 4), np.float32)
    d = np.zeros((1, 1, 4), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.verify_accept_stochastic(z, d, np.array([-1, 1]), np.array([0, 1]), np.array([0, 2]), 1,
                                        np.zeros(2), np.zeros(2))
    with pytest.raises(oracle.OracleError):
        oracle.verify_accept_stochastic(z, d, np.array([-1, 0]), np.array([0, 9]), np.array([0, 2]), 1,
                                        np.zeros(2), np.zeros(2))
