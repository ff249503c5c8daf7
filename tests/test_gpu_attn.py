"""GPU parity of jt_tree_attn_paged against the oracle.

bf16 in, fp32 accumulate: max abs error <= 2e-2 and mean abs error <= 2e-3
against the fp64 oracle (the task's stated tolerance); lse within 2e-2.
fp32 inputs (CUDA-core path): max abs <= 1e-4.  Trees come from the oracle's
build; every input from the seeded generators."""

import os

import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_jt_gb300 as jt
from tree_speculative_decoding_jt_gb300 import workloads as wk
from gpu_util import attn_errors, dev, kv_to_device, oracle_attn_threaded, oracle_tree, to_np_bf16

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, LSE_TOL, F32_MAX = 2e-2, 2e-3, 2e-2, 1e-4


# JT_ATTN_KERNEL=pair runs D = 128 on the CTA-pair kernel, "single" on the
# single-SM kernel (which D = 64 always uses).  Every parity case runs both.
KERNELS = ("pair", "single")


def _gpu(wl, tree, kernel):
    q, k, v = kv_to_device(wl)
    old = os.environ.get("JT_ATTN_KERNEL")
    os.environ["JT_ATTN_KERNEL"] = kernel
    try:
        out, lse = jt.jt_tree_attn_paged(q, k, v, dev(wl.block_table), dev(wl.prefix_len),
                                         dev(wl.tree_off), dev(tree["anc"].view(np.int32)),
                                         scale=wl.scale, max_tree=int(np.diff(wl.tree_off).max()))
        torch.cuda.synchronize()
    finally:
        if old is None:
            os.environ.pop("JT_ATTN_KERNEL", None)
        else:
            os.environ["JT_ATTN_KERNEL"] = old
    got = to_np_bf16(out) if out.dtype == torch.bfloat16 else out.cpu().numpy()
    return got, lse.cpu().numpy()


def _run(wl, tree, rows=None, threaded=False, kernels=KERNELS):
    """The library's output under each kernel choice, and the oracle's."""
    gots = []
    for kern in kernels:
        got, got_lse = _gpu(wl, tree, kern)
        if rows is not None:
            got, got_lse = got[rows], got_lse[rows]
        gots.append((got, got_lse))
    if threaded:
        want, want_lse = oracle_attn_threaded(wl, tree["parent"], rows)
    else:
        want, want_lse = oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.prefix_len,
                                          wl.tree_off, tree["parent"], wl.scale, rows=rows)
    return gots, want, want_lse


def _check_bf16(got, got_lse, want, want_lse):
    assert np.all(np.isfinite(got))
    mx, mean = attn_errors(got, want)
    assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)
    assert np.abs(got_lse - want_lse).max() <= LSE_TOL


def _check_all(gots, want, want_lse):
    for got, got_lse in gots:
        _check_bf16(got, got_lse, want, want_lse)


def _small(seed, nseq, Hq, Hkv, D, prefix, budgets, N=6, W=3, dtype="bf16", q_mult=None, poison=False):
    o = dict(dtype=dtype, nseq=nseq, Hq=Hq, Hkv=Hkv, D=D, prefix=("list", prefix), budgets=budgets,
             N=N, W=W, V=300, qkv_std=0.5 if dtype == "bf16" else 1.0)
    if q_mult:
        o["q_mult"] = q_mult
    return wk.make(2, seed=seed, overrides=o, poison=poison)


@pytest.mark.parametrize("case", [
    # seed, nseq, Hq, Hkv, D, prefix lengths, budgets
    (1, 1, 32, 8, 128, [300], (40,)),
    (2, 3, 32, 8, 128, [0, 1, 129], (1, 33, 100)),
    (3, 2, 32, 8, 128, [127, 128], (256, 64)),
    (4, 4, 32, 8, 128, [15, 16, 17, 1000], (5, 32, 31, 129)),
    (5, 2, 8, 8, 128, [200, 3], (70, 130)),        # G = 1
    (6, 2, 16, 8, 128, [64, 257], (48, 90)),       # G = 2
    (7, 2, 64, 8, 128, [100, 50], (20, 40)),       # G = 8
    (8, 2, 32, 8, 64, [500, 33], (77, 12)),        # D = 64
    (9, 1, 32, 2, 128, [2000], (256,)),            # G = 16: 16 query-tile pairs per KV head
    (10, 1, 32, 8, 128, [1500], (100,)),           # units cut into 1-2 tile pieces across CTAs
    (11, 1, 32, 8, 64, [900], (37,)),              # the same with D = 64
    (12, 1, 32, 8, 128, [700], (20,)),             # one query tile per unit (tile B absent)
    (13, 1, 32, 8, 128, [7000], (30,)),            # each unit merged from ~3 CTAs' partials
])
def test_bf16_matches_oracle_all_nodes(case):
    seed, nseq, Hq, Hkv, D, prefix, budgets = case
    wl = _small(seed, nseq, Hq, Hkv, D, prefix, budgets)
    tree = oracle_tree(wl)
    _check_all(*_run(wl, tree))


def test_bf16_deep_tree_long_ancestor_chains():
    """A tree about 64 deep (peaked draft rows: the top-1 log-prob near 0),
    so nodes see up to 65 tree keys through their ancestor sets."""
    wl = _small(21, 2, 32, 8, 128, [333, 64], (256, 200), N=64, W=2)
    wl.draft_logits[:] *= np.float32(40.0 / np.sqrt(2))
    tree = oracle_tree(wl)
    assert tree["depth"].max() >= 48
    _check_all(*_run(wl, tree))


def test_bf16_peaky_scores():
    """Q scaled by 8: softmax far from uniform, exercises the rescaling."""
    wl = _small(11, 2, 32, 8, 128, [700, 40], (96, 200), q_mult=8.0)
    _check_all(*_run(wl, oracle_tree(wl)))


def test_bf16_running_max_jumps_late():
    """q scaled by 8 and the keys of one late prefix page scaled by 20: at that
    tile the running maximum jumps by far more than 2^32 (log2 units), so both
    kernels must rescale O there (their lazy thresholds are 2^8 and 2^32)."""
    wl = _small(15, 2, 32, 8, 128, [1000, 2000], (40, 100), q_mult=8.0)
    for b in range(wl.nseq):
        pg = wl.block_table[b, (int(wl.prefix_len[b]) - 40) // 16]
        wl.k_cache[pg] = wk.f32_to_bf16_bits(wk.bf16_bits_to_f32(wl.k_cache[pg]) * np.float32(20.0))
    _check_all(*_run(wl, oracle_tree(wl)))


def test_bf16_poisoned_pool_is_never_read():
    """Spare pages and page tails past each tree hold NaN; a read outside
    the block table or past the last node would show up in the output."""
    wl = _small(12, 3, 32, 8, 128, [33, 250, 7], (17, 100, 256), poison=True)
    _check_all(*_run(wl, oracle_tree(wl)))


def test_bf16_sibling_kv_does_not_change_output():
    wl = _small(13, 1, 32, 8, 128, [130], (64,))
    tree = oracle_tree(wl)
    gots, *_ = _run(wl, tree)
    # overwrite the K/V of every tree slot that is not an ancestor-or-self of node 63
    n = 63
    anc = set()
    u = n
    while u >= 0:
        anc.add(u)
        u = tree["parent"][u]
    rng = np.random.default_rng(0)
    L = int(wl.prefix_len[0])
    for j in range(64):
        if j in anc:
            continue
        slot = L + j
        pg = wl.block_table[0, slot // 16]
        wl.k_cache[pg, slot % 16] = wk.f32_to_bf16_bits(rng.standard_normal((8, 128)) * 5)
        wl.v_cache[pg, slot % 16] = wk.f32_to_bf16_bits(rng.standard_normal((8, 128)) * 5)
    gots2, *_ = _run(wl, tree)
    for (got, _), (got2, _) in zip(gots, gots2):
        assert np.array_equal(got2[n], got[n])


def test_f32_config1_full():
    wl = wk.make(1)
    tree = oracle_tree(wl)
    [(got, got_lse)], want, want_lse = _run(wl, tree, kernels=("pair",))
    assert np.abs(got - want).max() <= F32_MAX
    assert np.abs(got_lse - want_lse).max() <= F32_MAX


def _whole_sequences(wl, seqs):
    """Every node of the listed sequences (global node indices)."""
    return np.concatenate([np.arange(wl.tree_off[b], wl.tree_off[b + 1], dtype=np.int32) for b in seqs])


def _longest(wl, candidates):
    return max(candidates, key=lambda b: (int(wl.prefix_len[b]), -b))


def test_bf16_drafter_tree_only_all_nodes():
    """The drafter-shaped workload: every node attends to its ancestors
    only (no prefix); all 16 x 256 nodes and 32 heads against the oracle."""
    wl = wk.make(6)
    tree = oracle_tree(wl)
    _check_all(*_run(wl, tree))


def test_bf16_config2_every_node():
    """Batch 1, prefix 4096, B = 256: all 256 nodes x 32 heads (the KV range
    is split over several CTAs and merged by the combine)."""
    wl = wk.make(2)
    tree = oracle_tree(wl)
    _check_all(*_run(wl, tree, rows=_whole_sequences(wl, [0]), threaded=True))


def test_bf16_config3_whole_sequences():
    """The ragged serving batch: every node and head of the longest-prefix
    sequence with B = 128 and of the longest-prefix one with B = 256."""
    wl = wk.make(3)
    tree = oracle_tree(wl)
    budgets = np.diff(wl.tree_off)
    seqs = [_longest(wl, [b for b in range(wl.nseq) if budgets[b] == 128]),
            _longest(wl, [b for b in range(wl.nseq) if budgets[b] == 256])]
    _check_all(*_run(wl, tree, rows=_whole_sequences(wl, seqs), threaded=True))


def test_bf16_config5_whole_sequences():
    """The verify-step batch (B = 256, prefixes 2k-16k): every node and head
    of the longest- and of the shortest-prefix sequence."""
    wl = wk.make(5)
    tree = oracle_tree(wl)
    order = np.argsort(wl.prefix_len, kind="stable")
    seqs = [int(order[-1]), int(order[0])]
    _check_all(*_run(wl, tree, rows=_whole_sequences(wl, seqs), threaded=True))


@pytest.mark.slow
def test_bf16_config4_whole_sequences():
    """32 sequences of prefix 32768, B = 64: all 64 nodes x 32 heads of the
    first and of the last sequence."""
    wl = wk.make(4)
    tree = oracle_tree(wl)
    _check_all(*_run(wl, tree, rows=_whole_sequences(wl, [0, wl.nseq - 1]), threaded=True))


def test_host_side_argument_errors():
    wl = _small(14, 1, 32, 8, 128, [1000], (4,))
    q, k, v = kv_to_device(wl)
    bt, pl, off = dev(wl.block_table), dev(wl.prefix_len), dev(wl.tree_off)
    anc = torch.zeros((4, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(jt.JtError) as e:   # D = 96 unsupported on the bf16 path
        jt.jt_tree_attn_paged(q[:, :, :96].contiguous(), k[..., :96].contiguous(),
                              v[..., :96].contiguous(), bt, pl, off, anc, max_tree=4)
    assert e.value.status == -2
    with pytest.raises(jt.JtError) as e:   # workspace too small for the plan and the partials
        jt.jt_tree_attn_paged(q, k, v, bt, pl, off, anc, max_tree=4, ws=jt.workspace(256))
    assert e.value.status == -5


@pytest.mark.parametrize("kernel", KERNELS)
def test_repeated_calls_on_one_workspace_and_stale_merge_counts(kernel, monkeypatch):
    """Units cut across work slots are merged by the slot that finishes last,
    counted in the workspace with the number of the call: repeated calls on
    one workspace give identical outputs, and counts left behind by an
    earlier call (planted here: call number 0 with a count of 7) are
    ignored."""
    monkeypatch.setenv("JT_ATTN_KERNEL", kernel)
    wl = _small(31, 2, 32, 8, 128, [2500, 900], (200, 64))
    tree = oracle_tree(wl)
    q, k, v = kv_to_device(wl)
    args = (q, k, v, dev(wl.block_table), dev(wl.prefix_len), dev(wl.tree_off), dev(tree["anc"].view(np.int32)))
    ws = jt.workspace(jt.jt_workspace_size(jt.JT_OP_TREE_ATTN, wl.nseq, 0, 0, 0, wl.total, 32, 8, 128,
                                           wl.block_table.shape[1], 200))
    outs = []
    for i in range(4):
        if i == 2:   # stale counts right after the header
            cnt = ws[256:256 + 16 * torch.cuda.get_device_properties(0).multi_processor_count].view(torch.int64)
            cnt.fill_(7)
        out, lse = jt.jt_tree_attn_paged(*args, scale=wl.scale, max_tree=200, ws=ws)
        jt.jt_check(ws)
        outs.append((to_np_bf16(out), lse.cpu().numpy()))
    for o, l in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1])
    want, want_lse = oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.prefix_len, wl.tree_off,
                                      tree["parent"], wl.scale)
    _check_bf16(outs[0][0], outs[0][1], want, want_lse)


def _attn_args(wl, tree):
    q, k, v = kv_to_device(wl)
    return (q, k, v, dev(wl.block_table), dev(wl.prefix_len), dev(wl.tree_off), dev(tree["anc"].view(np.int32)))


@pytest.mark.parametrize("kernel", KERNELS)
def test_calls_with_different_grids_share_one_workspace(kernel, monkeypatch):
    """A batch-1 call (split mode, a grid of its own) and a batch call (work-
    balanced, units cut across work slots) alternate on one workspace: every
    call of either kind numbers its merge counts consistently whatever the
    grid of the calls before it, so the outputs never change."""
    monkeypatch.setenv("JT_ATTN_KERNEL", kernel)
    wa = _small(41, 1, 32, 8, 128, [3000], (64,))
    wb = _small(42, 3, 32, 8, 128, [2500, 900, 4000], (200, 64, 150))
    ta, tb = oracle_tree(wa), oracle_tree(wb)
    aa, ab = _attn_args(wa, ta), _attn_args(wb, tb)
    size = max(jt.jt_workspace_size(jt.JT_OP_TREE_ATTN, w.nseq, 0, 0, 0, w.total, 32, 8, 128,
                                    w.block_table.shape[1], mt)
               for w, mt in ((wa, 64), (wb, 200)))
    ws = jt.workspace(size)
    outs_a, outs_b = [], []
    for _ in range(3):
        o, l = jt.jt_tree_attn_paged(*aa, scale=wa.scale, max_tree=64, ws=ws)
        jt.jt_check(ws)
        outs_a.append((to_np_bf16(o), l.cpu().numpy()))
        o, l = jt.jt_tree_attn_paged(*ab, scale=wb.scale, max_tree=200, ws=ws)
        jt.jt_check(ws)
        outs_b.append((to_np_bf16(o), l.cpu().numpy()))
    for outs, w, t in ((outs_a, wa, ta), (outs_b, wb, tb)):
        for o, l in outs[1:]:
            assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1])
        want, want_lse = oracle.tree_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.prefix_len, w.tree_off,
                                          t["parent"], w.scale)
        _check_bf16(outs[0][0], outs[0][1], want, want_lse)
