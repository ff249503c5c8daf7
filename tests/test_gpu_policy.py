"""GPU parity of the adaptive tree policy (AdaptiveSpec's per-step tree
policy) and of the width/depth-capped expansion against the oracle.

Integer outputs and the fp64 rolling average must be bit-identical: the
kernel rounds every fp64 operation the way the definition does.  For the
fused build (GPU top-W tables, whose log-probs differ from the oracle's by
~1e-12), requests whose confidence lies within 1e-9 of the threshold, or
trees with a decision gap below 1e-9, would be ambiguous and are ruled out
by construction of the inputs (asserted).  Attention and acceptance then run
over the device-written offsets with node arrays sized to the policy's
capacity; rows past the last tree must stay untouched."""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_jt_gb300 as jt
from tree_speculative_decoding_jt_gb300 import workloads as wk
from gpu_util import attn_errors, dev, kv_to_device, to_np_bf16

pytestmark = pytest.mark.gpu

AMBIGUOUS = 1e-9


def _tables(rng, nseq, N, W, ties=False):
    lp = -np.sort(rng.exponential(1.0, size=(nseq, N, W)), axis=2)
    if ties:
        lp = np.round(lp, 1)
    tok = np.stack([np.stack([np.sort(rng.choice(5000, size=W, replace=False)) for _ in range(N)])
                    for _ in range(nseq)]).astype(np.int32)
    return tok, lp


def _full(n, w):
    return sum(w ** d for d in range(n + 1))


def _oracle_params(p):
    return dict(b_min=p.b_min, b_max=p.b_max, node_cap=p.node_cap, w_min=p.w_min, n_min=p.n_min,
                n_slack=p.n_slack, beta=p.beta, log_conf=p.log_conf, acc_thresh=p.acc_thresh)


def _cmp_tree(got, want, hi):
    par, tk, dp, anc = (t.cpu().numpy() for t in got)
    np.testing.assert_array_equal(par[:hi], want["parent"])
    np.testing.assert_array_equal(tk[:hi], want["token"])
    np.testing.assert_array_equal(dp[:hi], want["depth"])
    np.testing.assert_array_equal(anc[:hi].view(np.uint32), want["anc"])


@pytest.mark.parametrize("seed", range(6))
def test_capped_expansion_bit_exact(seed):
    rng = np.random.default_rng(300 + seed)
    nseq, N, W = int(rng.integers(1, 12)), int(rng.integers(1, 10)), int(rng.integers(1, 9))
    tok, lp = _tables(rng, nseq, N, W, ties=bool(seed % 2))
    wc = rng.integers(1, W + 1, size=nseq).astype(np.int32)
    nc = rng.integers(0, N + 1, size=nseq).astype(np.int32)
    budgets = [int(rng.integers(1, min(_full(int(n), int(w)), 256) + 1)) for n, w in zip(nc, wc)]
    off = np.concatenate([[0], np.cumsum(budgets)]).astype(np.int32)
    root = rng.integers(0, 5000, size=nseq).astype(np.int32)
    want = oracle.tree_expand_capped(tok, lp, root, off, N, W, w_cap=wc, n_cap=nc)
    got = jt.jt_tree_expand_capped(dev(tok), dev(lp), dev(root), dev(off), dev(wc), dev(nc),
                                   total_nodes=int(off[-1]) + 17)      # capacity above the total
    torch.cuda.synchronize()
    _cmp_tree(got, want, int(off[-1]))


def test_capped_expansion_one_cap_only_and_bad_caps():
    rng = np.random.default_rng(9)
    tok, lp = _tables(rng, 2, 5, 4)
    root = np.array([1, 2], np.int32)
    off = np.array([0, 6, 12], np.int32)
    for kw in (dict(n_cap=np.array([2, 5], np.int32)), dict(w_cap=np.array([1, 2], np.int32))):
        want = oracle.tree_expand_capped(tok, lp, root, off, 5, 4, **kw)
        got = jt.jt_tree_expand_capped(dev(tok), dev(lp), dev(root), dev(off),
                                       **{k: dev(v) for k, v in kw.items()})
        torch.cuda.synchronize()
        _cmp_tree(got, want, 12)
    ws = jt.workspace(256)
    jt.jt_tree_expand_capped(dev(tok), dev(lp), dev(root), dev(off), w_cap=dev(np.array([1, 5], np.int32)),
                             ws=ws)                                # 5 > W
    with pytest.raises(jt.JtError):
        jt.jt_check(ws)
    jt.jt_tree_expand_capped(dev(tok), dev(lp), dev(root), dev(off), n_cap=dev(np.array([1, 1], np.int32)),
                             ws=ws)                                # 6 > full(1, 4) = 5
    with pytest.raises(jt.JtError):
        jt.jt_check(ws)


@pytest.mark.parametrize("nseq,node_cap", [(5, 0), (1024, 0), (3000, 40000), (70, 900)])
def test_policy_kernel_bit_exact_over_steps(nseq, node_cap):
    rng = np.random.default_rng(nseq + node_cap)
    N, W = 8, 4
    prm = jt.policy_params(b_min=4, b_max=200, node_cap=node_cap, w_min=2, n_min=1, n_slack=2, beta=0.3,
                           log_conf=float(np.log(0.55)), acc_thresh=2.5)
    bs = rng.integers(1, 300, size=nseq).astype(np.int32)
    ema = rng.uniform(0, N, size=nseq)
    bs_d, ema_d = dev(bs), dev(ema)
    acc = None
    for step in range(6):
        lp = -np.sort(rng.exponential(0.8, size=(nseq, N, W)), axis=2)
        want = oracle.tree_policy(lp, acc, bs, ema, **_oracle_params(prm))
        off, wc, nc = jt.jt_tree_policy(dev(lp), None if acc is None else dev(acc), bs_d, ema_d, prm)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(off.cpu().numpy(), want["tree_off"])
        np.testing.assert_array_equal(wc.cpu().numpy(), want["w_cap"])
        np.testing.assert_array_equal(nc.cpu().numpy(), want["n_cap"])
        np.testing.assert_array_equal(bs_d.cpu().numpy(), want["budget_state"])
        np.testing.assert_array_equal(ema_d.cpu().numpy(), want["acc_ema"])      # bit-identical fp64
        bs, ema = want["budget_state"], want["acc_ema"]
        acc = rng.integers(-1, N + 1, size=nseq).astype(np.int32)


def test_policy_invalid_state_gives_root_only_tree():
    N, W = 4, 2
    lp = dev(np.full((3, N, W), -0.1))
    bs = dev(np.array([16, 16, 16], np.int32))
    ema = dev(np.array([1.0, -1.0, 2.0]))
    acc = dev(np.array([2, 1, N + 1], np.int32))
    ws = jt.workspace(256)
    off, wc, nc = jt.jt_tree_policy(lp, acc, bs, ema, jt.policy_params(b_min=2, w_min=1, n_min=0), ws=ws)
    with pytest.raises(jt.JtError) as e:
        jt.jt_check(ws)
    assert e.value.status == -1
    b = np.diff(off.cpu().numpy())
    assert b[1] == 1 and b[2] == 1 and b[0] > 1
    assert list(nc.cpu().numpy()[1:]) == [0, 0]
    np.testing.assert_array_equal(ema.cpu().numpy()[1:], [-1.0, 2.0])      # state left as it was
    np.testing.assert_array_equal(bs.cpu().numpy()[1:], [16, 16])


def _adaptive_case(seed, nseq, N, W, V):
    wl = wk.make(1, seed=seed, overrides=dict(dtype="f32", nseq=nseq, Hq=4, Hkv=1, D=64, prefix=("fixed", 0),
                                             budgets=(1,), N=N, W=W, V=V, qkv_std=1.0))
    return wl.draft_logits, wl.root_token


@pytest.mark.parametrize("seed", range(3))
def test_adaptive_build_matches_oracle_over_steps(seed):
    """topw -> policy -> capped expansion fused on the GPU against the
    oracle's tree_build tables -> tree_policy -> tree_expand_capped."""
    rng = np.random.default_rng(400 + seed)
    nseq, N, W, V = 12, 6, 3, 2000
    prm = jt.policy_params(b_min=4, b_max=128, w_min=1, n_min=1, n_slack=2, beta=0.5, acc_thresh=2.0,
                           log_conf=float(np.log(0.3)))
    cap = nseq * jt.policy_ceiling(prm, nseq)
    bs = np.full(nseq, 16, np.int32)
    ema = np.full(nseq, 2.0)
    bs_d, ema_d = dev(bs), dev(ema)
    acc = None
    for step in range(4):
        z, root = _adaptive_case(1000 * seed + step, nseq, N, W, V)
        z = z * rng.uniform(0.5, 6.0, size=(nseq, 1, 1)).astype(np.float32)   # spread of confidences
        tb = oracle.tree_build(z, root, np.arange(nseq + 1, dtype=np.int32), W)
        assert np.min(np.abs(tb["lp"][:, 0, 0] - prm.log_conf)) > AMBIGUOUS
        pol = oracle.tree_policy(tb["lp"], acc, bs, ema, **_oracle_params(prm))
        want = oracle.tree_expand_capped(tb["tok"], tb["lp"], root, pol["tree_off"], N, W,
                                         w_cap=pol["w_cap"], n_cap=pol["n_cap"])
        assert np.min(want["gap"]) > AMBIGUOUS
        out = jt.jt_tree_build_adaptive(dev(z), dev(root), None if acc is None else dev(acc), bs_d, ema_d, W,
                                        prm, capacity=cap)
        torch.cuda.synchronize()
        off, wc, nc = (t.cpu().numpy() for t in out[:3])
        np.testing.assert_array_equal(off, pol["tree_off"])
        np.testing.assert_array_equal(wc, pol["w_cap"])
        np.testing.assert_array_equal(nc, pol["n_cap"])
        np.testing.assert_array_equal(bs_d.cpu().numpy(), pol["budget_state"])
        np.testing.assert_array_equal(ema_d.cpu().numpy(), pol["acc_ema"])
        _cmp_tree(out[3:], want, int(off[-1]))
        bs, ema = pol["budget_state"], pol["acc_ema"]
        acc = rng.integers(0, N + 1, size=nseq).astype(np.int32)


def test_attention_and_acceptance_over_device_offsets_with_spare_capacity():
    """The adaptive build's offsets feed jt_tree_attn_paged (bf16, units cut across CTAs)
    and jt_verify_accept with total_nodes = capacity: the trees' rows match
    the oracle and the spare rows past the last tree are never written."""
    nseq, N, W, V = 3, 6, 3, 500
    prm = jt.policy_params(b_min=8, b_max=64, w_min=2, n_min=2, n_slack=2)
    ceil_b = jt.policy_ceiling(prm, nseq)
    cap = nseq * ceil_b
    wl = wk.make(2, seed=77, overrides=dict(dtype="bf16", nseq=nseq, Hq=32, Hkv=8, D=128,
                                            prefix=("list", [900, 40, 333]), budgets=(ceil_b,), N=N, W=W,
                                            V=V, qkv_std=0.5))
    assert wl.total == cap
    bs = dev(np.array([64, 8, 30], np.int32))
    ema = dev(np.array([5.0, 0.0, 2.0]))
    z = wl.draft_logits.copy()
    z[0] *= 8.0                        # confident first request
    off, wc, nc, parent, token, depth, anc = jt.jt_tree_build_adaptive(
        dev(z), dev(wl.root_token), None, bs, ema, W, prm, capacity=cap)
    torch.cuda.synchronize()
    off_h = off.cpu().numpy()
    total = int(off_h[-1])
    assert total < cap
    q, k, v = kv_to_device(wl)
    out = torch.full((cap, 32, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((cap, 32), 7.0, dtype=torch.float32, device="cuda")
    jt.jt_tree_attn_paged(q, k, v, dev(wl.block_table), dev(wl.prefix_len), off, anc, scale=wl.scale,
                          max_tree=ceil_b, out=out, lse=lse)
    torch.cuda.synchronize()
    par_h = parent.cpu().numpy()[:total]
    want, want_lse = oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.prefix_len, off_h,
                                      par_h, wl.scale, rows=np.arange(total, dtype=np.int32))
    got = to_np_bf16(out)
    mx, mean = attn_errors(got[:total], want)
    assert mx <= 2e-2 and mean <= 2e-3, (mx, mean)
    assert np.abs(lse.cpu().numpy()[:total] - want_lse).max() <= 2e-2
    assert np.all(got[total:] == 7.0) and np.all(lse.cpu().numpy()[total:] == 7.0)
    # acceptance over the same device offsets
    rng = np.random.default_rng(5)
    target = (rng.standard_normal((cap, V)) * np.sqrt(2)).astype(np.float32)
    tok_h = token.cpu().numpy()
    for bq in range(nseq):      # boost most drafted tokens in their parent's row: long paths occur
        for c in range(off_h[bq] + 1, off_h[bq + 1]):
            if rng.random() < 0.8:
                row = off_h[bq] + par_h[c]
                target[row, tok_h[c]] = target[row].max() + 1.0
    acc, path, bonus = jt.jt_verify_accept(dev(target), parent, token, off, N, rule=jt.JT_RULE_GREEDY)
    torch.cuda.synchronize()
    wa, wp, wb = oracle.verify_accept(target[:total], par_h, token.cpu().numpy()[:total], off_h, N, 0)
    np.testing.assert_array_equal(acc.cpu().numpy(), wa)
    np.testing.assert_array_equal(path.cpu().numpy(), wp)
    np.testing.assert_array_equal(bonus.cpu().numpy(), wb)
