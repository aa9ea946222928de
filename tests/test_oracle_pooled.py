"""Pins for the GQA-pooled index sets of oracle/attention.py.

Pooled mode keeps one set per (sequence, KV head): key j's score is the sum
over the group's query heads of their post-softmax weights (decode) or tile
weights (prefill). What fixes it independently of its own code:

* invariants: each group's decode weights sum to its number of heads, its
  tile weights to heads x rows of the tile (every softmax row sums to 1);
* reductions: with one query head per KV head the pooled sets are the
  per-head sets; when a group's heads share one query the pooled set is
  that query's per-head set;
* the group map: heads planted on distinct keys put exactly their own keys
  into their own group's set, under a permuted map;
* reuse: equals the library SDPA routine with a mask holding each head's
  group set; k = N is dense; NaN outside the group sets changes nothing;
* prefill tiles whose prefix fits in k select the whole prefix.
"""
import math

import numpy as np
import torch
import torch.nn.functional as F

from oracle import attention as A
from oracle.topk import topk_indices


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _sdpa(q, k, v, mask=None, causal=False, scale=None):
    return F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                          torch.from_numpy(v),
                                          attn_mask=None if mask is None else torch.from_numpy(mask),
                                          is_causal=causal, scale=scale).numpy()


def test_pooled_decode_weights_sum_to_group_size():
    rng = np.random.default_rng(101)
    B, Hq, Hkv, N, d = 2, 6, 2, 45, 8
    gmap = [1, 0, 1, 0, 0, 1]
    q, K, V = _rand(rng, B, Hq, d), 3 * _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    _, idx, w = A.anchor_decode_pooled(q, K, V, 7, gmap, 0.5)
    assert w.shape == (B, Hkv, N) and idx.shape == (B, Hkv, 7)
    np.testing.assert_allclose(w.sum(-1), 3.0, atol=1e-12)
    assert (w >= 0).all() and (w <= 3.0).all()
    for b in range(B):
        for g in range(Hkv):
            assert idx[b, g].tolist() == topk_indices(w[b, g], 7).tolist()


def test_pooled_decode_one_head_per_group_is_per_head():
    rng = np.random.default_rng(102)
    B, H, N, d, k = 2, 3, 80, 8, 11
    q, K, V = _rand(rng, B, H, d), _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    o_p, idx_p, w = A.anchor_decode_pooled(q, K, V, k)
    o_h, idx_h, s = A.anchor_decode(q, K, V, k)
    assert (idx_p == idx_h).all()
    np.testing.assert_array_equal(o_p, o_h)
    np.testing.assert_allclose(w, A.softmax(s), atol=1e-15)


def test_pooled_decode_shared_query_is_per_head_set():
    rng = np.random.default_rng(103)
    B, Hq, Hkv, N, d, k = 1, 4, 1, 64, 8, 9
    q1 = _rand(rng, B, 1, d)
    q = np.repeat(q1, Hq, axis=1)
    K, V = _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    _, idx_p, w = A.anchor_decode_pooled(q, K, V, k)
    _, idx_h, s = A.anchor_decode(q, K, V, k)
    for h in range(Hq):
        assert idx_p[0, 0].tolist() == idx_h[0, h].tolist()
    np.testing.assert_allclose(w[0, 0], Hq * A.softmax(s[0, 0]), atol=1e-13)


def test_pooled_decode_follows_the_group_map():
    # head h's query points at key 10 + h only; its group's set must hold
    # exactly the keys of the heads mapped to it
    B, Hq, Hkv, N, d = 1, 6, 3, 40, 16
    gmap = [2, 0, 1, 1, 2, 0]
    K = np.zeros((B, Hkv, N, d))
    q = np.zeros((B, Hq, d))
    for h in range(Hq):
        q[0, h, h] = 30.0
        K[0, gmap[h], 10 + h, h] = 1.0
    V = np.zeros((B, Hkv, N, d))
    _, idx, w = A.anchor_decode_pooled(q, K, V, 2, gmap, 1.0)
    for g in range(Hkv):
        want = sorted(10 + h for h in range(Hq) if gmap[h] == g)
        assert idx[0, g].tolist() == want
        for h in range(Hq):
            if gmap[h] == g:
                assert w[0, g, 10 + h] > 0.99


def test_pooled_sparse_decode_matches_masked_sdpa():
    rng = np.random.default_rng(104)
    B, Hq, Hkv, N, d, k = 2, 6, 2, 50, 8, 9
    gmap = [0, 1, 1, 0, 1, 0]
    q, K, V = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    idx = np.stack([np.stack([np.sort(rng.choice(N, k, replace=False)) for _ in range(Hkv)])
                    for _ in range(B)])
    o = A.sparse_decode_pooled(q, K, V, idx, gmap, 0.4)
    mask = np.zeros((B, Hq, 1, N), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            mask[b, h, 0, idx[b, gmap[h]]] = True
    ref = _sdpa(q[:, :, None, :], K[:, gmap], V[:, gmap], mask=mask, scale=0.4)[:, :, 0]
    np.testing.assert_allclose(o, ref, atol=1e-12)


def test_pooled_sparse_decode_k_equals_n_and_poison():
    rng = np.random.default_rng(105)
    B, Hq, Hkv, N, d = 1, 4, 2, 30, 8
    q, K, V = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    o_d, idx, _ = A.anchor_decode_pooled(q, K, V, N)
    np.testing.assert_allclose(A.sparse_decode_pooled(q, K, V, idx), o_d, atol=1e-13)
    _, idx, _ = A.anchor_decode_pooled(q, K, V, 5)
    o = A.sparse_decode_pooled(q, K, V, idx)
    Kp, Vp = K.copy(), V.copy()
    for g in range(Hkv):
        out = np.setdiff1d(np.arange(N), idx[0, g])
        Kp[0, g, out] = np.nan
        Vp[0, g, out] = np.nan
    np.testing.assert_array_equal(A.sparse_decode_pooled(q, Kp, Vp, idx), o)


def test_pooled_tile_weights_sum_and_one_head_reduction():
    rng = np.random.default_rng(106)
    B, Hq, Hkv, N, d = 1, 4, 2, 300, 8
    gmap = [1, 0, 0, 1]
    Q, K = _rand(rng, B, Hq, N, d), _rand(rng, B, Hkv, N, d)
    for t in range(A.n_tiles(N)):
        r0, r1 = A.tile_rows(t, N)
        for g in range(Hkv):
            w = A.tile_weights_pooled(Q, K, 0, g, t, gmap, 0.35)
            assert w.shape == (A.prefix_len(t, N),)
            np.testing.assert_allclose(w.sum(), 2 * (r1 - r0), atol=1e-10)
    # one query head per KV head: pooled tile sets are the per-head ones
    Q1, K1, V1 = _rand(rng, 1, 2, 260, 8), _rand(rng, 1, 2, 260, 8), _rand(rng, 1, 2, 260, 8)
    _, idx_p = A.anchor_prefill_pooled(Q1, K1, V1, 70)
    _, idx_h = A.anchor_prefill(Q1, K1, V1, 70)
    assert (idx_p == idx_h).all()


def test_pooled_prefill_prefix_tiles_and_reuse():
    rng = np.random.default_rng(107)
    B, Hq, Hkv, N, d, k = 1, 4, 2, 384, 8, 256
    gmap = [0, 1, 0, 1]
    Q, K, V = _rand(rng, B, Hq, N, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    o_a, idx = A.anchor_prefill_pooled(Q, K, V, k, gmap)
    assert idx.shape == (B, Hkv, 3, k)
    assert (idx[0, :, 0, :128] == np.arange(128)).all() and (idx[0, :, 0, 128:] == -1).all()
    assert (idx[0, :, 1] == np.arange(256)).all()
    assert (idx[0, :, 2] >= 0).all() and (np.diff(idx[0, :, 2], axis=-1) > 0).all()
    o_r = A.sparse_prefill_pooled(Q, K, V, idx, gmap)
    np.testing.assert_allclose(o_r[:, :, :256], o_a[:, :, :256], atol=1e-12)
    # the reuse rows of tile 2 equal the library routine with the group sets as the mask
    mask = np.zeros((B, Hq, N, N), dtype=bool)
    for h in range(Hq):
        for t in range(A.n_tiles(N)):
            sel = idx[0, gmap[h], t]
            sel = sel[sel >= 0]
            r0, r1 = A.tile_rows(t, N)
            for i in range(r0, r1):
                mask[0, h, i, sel[sel <= i]] = True
    ref = _sdpa(Q, K[:, gmap], V[:, gmap], mask=mask, scale=1 / math.sqrt(d))
    np.testing.assert_allclose(o_r, ref, atol=1e-12)
