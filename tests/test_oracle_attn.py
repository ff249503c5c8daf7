"""Pins for the oracle's tree-causal paged attention (CPU only).

Each check compares the oracle against something other than itself:
torch's scaled_dot_product_attention (a library routine) on explicit key
lists or with a causal mask, invariances the mask definition implies, and a
closed form.  Mask definition (JetSpec summary, tree-causal attention mask
paragraph; "加速AI思考…" section 三): a node sees the prefix and its own
ancestors (itself included), never siblings or descendants.
"""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_decoding_jt_gb300 import workloads as wk


def _sdpa(q, k, v, scale, mask=None):
    """torch SDPA in float64: q [H, n, D], k/v [H, m, D]."""
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=None if mask is None else torch.from_numpy(mask)[None, None],
        scale=scale)
    return out[0].numpy()


def _as_f64(a):
    return wk.bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def _gather_slots(cache, block_table, b, slots, page):
    pages = block_table[b, np.asarray(slots) // page]
    return cache[pages, np.asarray(slots) % page]  # [n, Hkv, D]


def _tiny(dtype="f32", **kw):
    o = dict(dtype=dtype, nseq=2, Hq=4, Hkv=2, D=16, prefix=("list", [37, 5]), budgets=(9, 6),
             N=3, W=2, V=50, qkv_std=1.0)
    o.update(kw)
    return wk.make(1, seed=7, overrides=o)


def _random_tree(rng, B):
    parent = np.full(B, -1, np.int32)
    for n in range(1, B):
        parent[n] = rng.integers(0, n)
    return parent


def _ancestor_path(parent, off, i):
    path = []
    u = i
    while u >= 0:
        path.append(u)
        u = parent[off + u]
    return path[::-1]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_each_node_equals_sdpa_over_its_explicit_key_list(dtype):
    wl = _tiny(dtype)
    rng = np.random.default_rng(3)
    parent = np.concatenate([_random_tree(rng, 9), _random_tree(rng, 6)])
    out, lse = oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.prefix_len,
                                wl.tree_off, parent, wl.scale)
    q, k, v = _as_f64(wl.q), _as_f64(wl.k_cache), _as_f64(wl.v_cache)
    G = 2
    for b in range(2):
        off, L = int(wl.tree_off[b]), int(wl.prefix_len[b])
        for i in range(int(wl.tree_off[b + 1]) - off):
            slots = list(range(L)) + [L + a for a in _ancestor_path(parent, off, i)]
            ks = _gather_slots(k, wl.block_table, b, slots, 16)  # [m, Hkv, D]
            vs = _gather_slots(v, wl.block_table, b, slots, 16)
            kh = np.repeat(ks.transpose(1, 0, 2), G, axis=0)     # head h -> kv head h // G
            vh = np.repeat(vs.transpose(1, 0, 2), G, axis=0)
            ref = _sdpa(q[off + i][:, None, :], kh, vh, wl.scale)[:, 0, :]
            np.testing.assert_allclose(out[off + i], ref, rtol=0, atol=1e-12)
            s = np.einsum("hd,hmd->hm", q[off + i], kh) * wl.scale
            np.testing.assert_allclose(lse[off + i], np.log(np.exp(s).sum(axis=1)), atol=1e-12)


def test_w1_chain_equals_causal_attention():
    """A chain tree (W=1) is ordinary causal attention: the i-th tree token
    at absolute position L+i attends to positions 0..L+i."""
    L, B, H, D = 45, 12, 3, 32
    o = dict(dtype="f32", nseq=1, Hq=H, Hkv=H, D=D, prefix=("list", [L]), budgets=(B,), N=B,
             W=1, V=20, qkv_std=1.0)
    wl = wk.make(1, seed=11, overrides=o)
    parent = np.arange(-1, B - 1, dtype=np.int32)
    out, _ = oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.prefix_len,
                              wl.tree_off, parent, wl.scale)
    slots = np.arange(L + B)
    k = _gather_slots(wl.k_cache.astype(np.float64), wl.block_table, 0, slots, 16).transpose(1, 0, 2)
    v = _gather_slots(wl.v_cache.astype(np.float64), wl.block_table, 0, slots, 16).transpose(1, 0, 2)
    qpos = L + np.arange(B)
    mask = slots[None, :] <= qpos[:, None]
    ref = _sdpa(wl.q.astype(np.float64).transpose(1, 0, 2), k, v, wl.scale, mask)
    np.testing.assert_allclose(out, ref.transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_sibling_and_descendant_kv_do_not_matter():
    wl = _tiny("bf16")
    rng = np.random.default_rng(4)
    parent = np.concatenate([_random_tree(rng, 9), _random_tree(rng, 6)])
    base, base_lse = oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                                      wl.prefix_len, wl.tree_off, parent, wl.scale)
    for b in range(2):
        off, L = int(wl.tree_off[b]), int(wl.prefix_len[b])
        Bb = int(wl.tree_off[b + 1]) - off
        for i in range(Bb):
            anc = set(_ancestor_path(parent, off, i))
            others = [j for j in range(Bb) if j not in anc]
            if not others:
                continue
            k2, v2 = wl.k_cache.copy(), wl.v_cache.copy()
            for j in others:
                slot = L + j
                pg = wl.block_table[b, slot // 16]
                k2[pg, slot % 16] = wk.f32_to_bf16_bits(rng.standard_normal(k2.shape[2:]) * 9)
                v2[pg, slot % 16] = wk.f32_to_bf16_bits(rng.standard_normal(v2.shape[2:]) * 9)
            out, lse = oracle.tree_attn(wl.q, k2, v2, wl.block_table, wl.prefix_len, wl.tree_off,
                                        parent, wl.scale, rows=[off + i])
            assert np.array_equal(out[0], base[off + i]) and np.array_equal(lse[0], base_lse[off + i])
            # ... while changing an ancestor's K does change it
            a = max(anc)
            k3 = wl.k_cache.copy()
            slot = L + a
            pg = wl.block_table[b, slot // 16]
            k3[pg, slot % 16] = wk.f32_to_bf16_bits(rng.standard_normal(k3.shape[2:]) * 9)
            out3, _ = oracle.tree_attn(wl.q, k3, wl.v_cache, wl.block_table, wl.prefix_len,
                                       wl.tree_off, parent, wl.scale, rows=[off + i])
            assert not np.array_equal(out3[0], base[off + i])


def test_page_permutation_leaves_output_unchanged():
    wl = _tiny("f32")
    parent = np.concatenate([_random_tree(np.random.default_rng(5), 9),
                             _random_tree(np.random.default_rng(6), 6)])
    base, _ = oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.prefix_len,
                               wl.tree_off, parent, wl.scale)
    perm = np.random.default_rng(8).permutation(wl.k_cache.shape[0])
    inv = np.argsort(perm)
    k2, v2 = wl.k_cache[perm], wl.v_cache[perm]          # physical page p moves to inv[p]
    bt2 = np.where(wl.block_table >= 0, inv[np.maximum(wl.block_table, 0)], -1)
    out, _ = oracle.tree_attn(wl.q, k2, v2, bt2, wl.prefix_len, wl.tree_off, parent, wl.scale)
    assert np.array_equal(out, base)


def test_constant_keys_closed_form_mean_of_visible_values():
    """With every key equal, the softmax is uniform over the visible keys,
    so each output is the plain mean of the visible V rows."""
    wl = _tiny("f32")
    k = np.ones_like(wl.k_cache)
    rng = np.random.default_rng(12)
    parent = np.concatenate([_random_tree(rng, 9), _random_tree(rng, 6)])
    out, lse = oracle.tree_attn(wl.q, k, wl.v_cache, wl.block_table, wl.prefix_len, wl.tree_off,
                                parent, wl.scale)
    for b in range(2):
        off, L = int(wl.tree_off[b]), int(wl.prefix_len[b])
        for i in range(int(wl.tree_off[b + 1]) - off):
            slots = list(range(L)) + [L + a for a in _ancestor_path(parent, off, i)]
            vs = _gather_slots(wl.v_cache.astype(np.float64), wl.block_table, b, slots, 16)
            mean = vs.mean(axis=0)                       # [Hkv, D]
            np.testing.assert_allclose(out[off + i], np.repeat(mean, 2, axis=0), atol=1e-12)
            s = wl.q[off + i].astype(np.float64).sum(axis=1) * wl.scale   # q . 1
            np.testing.assert_allclose(lse[off + i], s + np.log(len(slots)), atol=1e-12)


def test_empty_prefix_is_pure_tree_attention():
    wl = _tiny("f32", prefix=("list", [0, 0]))
    rng = np.random.default_rng(13)
    parent = np.concatenate([_random_tree(rng, 9), _random_tree(rng, 6)])
    out, _ = oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.prefix_len,
                              wl.tree_off, parent, wl.scale)
    # the root sees only itself: output = its own V row, broadcast over the group
    for b in range(2):
        off = int(wl.tree_off[b])
        pg = wl.block_table[b, 0]
        np.testing.assert_allclose(out[off], np.repeat(wl.v_cache[pg, 0].astype(np.float64), 2, 0),
                                   atol=1e-15)


def test_block_table_too_short_is_rejected():
    wl = _tiny("f32")
    parent = np.concatenate([_random_tree(np.random.default_rng(1), 9),
                             _random_tree(np.random.default_rng(2), 6)])
    with pytest.raises(oracle.OracleError):
        oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table[:, :1], wl.prefix_len,
                         wl.tree_off, parent, wl.scale)
