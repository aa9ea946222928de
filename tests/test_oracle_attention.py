"""Pins for oracle/attention.py.

* Dense decode / prefill equal torch's scaled_dot_product_attention run on
  the CPU in float64 (a library routine), including a permuted GQA map.
* Sparse (reuse) attention equals the same library routine with a boolean
  mask that keeps only the saved set (and the causal part in prefill).
* Closed forms: one key gives o = v; equal logits give the mean of V; two
  keys give the logistic weight.
* Invariants: softmax rows sum to 1; k = N makes sparse equal dense; NaN in
  every unselected K/V row leaves the sparse output bit-identical; a selected
  row changes it; prefill rows ignore future keys; tile weights sum to the
  number of rows in the tile; a one-row tile's weights are that row's
  probabilities; brute-force loops agree with the vectorised tile weights.
"""
import math

import numpy as np
import pytest
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


GMAPS = {"contiguous": [0, 0, 0, 1, 1, 1], "permuted": [1, 0, 1, 0, 0, 1]}


@pytest.mark.parametrize("gname", list(GMAPS))
def test_dense_decode_matches_sdpa(gname):
    rng = np.random.default_rng(1)
    B, Hq, Hkv, N, d = 2, 6, 2, 37, 16
    gmap = GMAPS[gname]
    q, K, V = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    o, s = A.dense_decode(q, K, V, gmap, 0.3)
    Kx = K[:, gmap]                       # [B, Hq, N, d]
    Vx = V[:, gmap]
    ref = _sdpa(q[:, :, None, :], Kx, Vx, scale=0.3)[:, :, 0]
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s, 0.3 * np.einsum("bhd,bhnd->bhn", q, Kx), atol=1e-12)


def test_default_scale_and_map():
    rng = np.random.default_rng(2)
    q, K, V = _rand(rng, 1, 4, 8), _rand(rng, 1, 2, 10, 8), _rand(rng, 1, 2, 10, 8)
    o, _ = A.dense_decode(q, K, V)
    o2, _ = A.dense_decode(q, K, V, [0, 0, 1, 1], 1 / math.sqrt(8))
    np.testing.assert_array_equal(o, o2)


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(3)
    p = A.softmax(50 * _rand(rng, 7, 300))
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
    assert (p >= 0).all()


def test_closed_forms():
    # one key: o = v exactly
    q = np.array([[[0.3, -1.0]]])
    K = np.array([[[[2.0, 5.0]]]])
    V = np.array([[[[7.0, -3.0]]]])
    o, _ = A.dense_decode(q, K, V, [0], 1.0)
    np.testing.assert_array_equal(o[0, 0], [7.0, -3.0])
    # equal logits: mean of V
    K = np.zeros((1, 1, 5, 2))
    V = np.arange(10.0).reshape(1, 1, 5, 2)
    o, _ = A.dense_decode(q, K, V, [0], 1.0)
    np.testing.assert_allclose(o[0, 0], V[0, 0].mean(0), atol=1e-15)
    # two keys: weight of key 0 is the logistic function of the logit gap
    q = np.array([[[1.0, 0.0]]])
    K = np.array([[[[1.5, 0.0], [0.0, 9.0]]]])
    V = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    o, s = A.dense_decode(q, K, V, [0], 0.5)
    w0 = 1.0 / (1.0 + math.exp(-(0.5 * 1.5 - 0.0)))
    np.testing.assert_allclose(o[0, 0], [w0, 1 - w0], atol=1e-15)
    np.testing.assert_allclose(s[0, 0], [0.75, 0.0], atol=1e-15)


def test_sparse_decode_matches_masked_sdpa():
    rng = np.random.default_rng(4)
    B, Hq, Hkv, N, d, k = 2, 4, 2, 50, 8, 9
    gmap = [0, 1, 1, 0]
    q, K, V = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    idx = np.stack([np.stack([np.sort(rng.choice(N, k, replace=False)) for _ in range(Hq)])
                    for _ in range(B)])
    o = A.sparse_decode(q, K, V, idx, gmap, 0.4)
    mask = np.zeros((B, Hq, 1, N), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            mask[b, h, 0, idx[b, h]] = True
    ref = _sdpa(q[:, :, None, :], K[:, gmap], V[:, gmap], mask=mask, scale=0.4)[:, :, 0]
    np.testing.assert_allclose(o, ref, atol=1e-12)


def test_k_equals_n_sparse_is_dense():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, N, d = 1, 4, 2, 33, 8
    q, K, V = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    o_a, idx, _ = A.anchor_decode(q, K, V, N)
    assert (idx == np.arange(N)).all()
    o_s = A.sparse_decode(q, K, V, idx)
    np.testing.assert_allclose(o_s, o_a, atol=1e-13)


def test_poison_and_perturbation():
    rng = np.random.default_rng(6)
    B, Hq, Hkv, N, d, k = 1, 2, 1, 40, 8, 6
    q, K, V = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    _, idx, _ = A.anchor_decode(q, K, V, k)
    o = A.sparse_decode(q, K, V, idx)
    sel = set(idx[0].ravel().tolist())
    Kp, Vp = K.copy(), V.copy()
    for j in range(N):
        if j not in sel:
            Kp[0, 0, j] = np.nan
            Vp[0, 0, j] = np.nan
    np.testing.assert_array_equal(A.sparse_decode(q, Kp, Vp, idx), o)
    j0 = int(idx[0, 0, 0])
    Vp = V.copy()
    Vp[0, 0, j0] += 1.0
    assert not np.array_equal(A.sparse_decode(q, K, Vp, idx)[0, 0], o[0, 0])


def test_anchor_decode_topk_of_logits_is_topk_of_probabilities():
    rng = np.random.default_rng(7)
    q, K, V = _rand(rng, 1, 2, 8), _rand(rng, 1, 1, 64, 8), _rand(rng, 1, 1, 64, 8)
    _, idx, s = A.anchor_decode(q, K, V, 10)
    p = A.softmax(s)
    for h in range(2):
        assert topk_indices(p[0, h], 10).tolist() == idx[0, h].tolist()


# ---------------------------------------------------------------- prefill --

@pytest.mark.parametrize("N", [128, 300])
def test_dense_prefill_matches_causal_sdpa(N):
    rng = np.random.default_rng(8)
    B, Hq, Hkv, d = 1, 4, 2, 16
    gmap = [1, 0, 0, 1]
    Q, K, V = _rand(rng, B, Hq, N, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    o = A.dense_prefill(Q, K, V, gmap, 0.25)
    ref = _sdpa(Q, K[:, gmap], V[:, gmap], causal=True, scale=0.25)
    np.testing.assert_allclose(o, ref, atol=1e-12)


def test_prefill_lse_closed_form():
    rng = np.random.default_rng(9)
    Q, K, V = _rand(rng, 1, 1, 200, 8), _rand(rng, 1, 1, 200, 8), _rand(rng, 1, 1, 200, 8)
    _, lse = A.dense_prefill_tile(Q, K, V, 0, 0, 1, [0], 0.5)
    for r, i in enumerate(range(128, 200)):
        s = 0.5 * K[0, 0, : i + 1] @ Q[0, 0, i]
        np.testing.assert_allclose(lse[r], math.log(np.exp(s).sum()), atol=1e-12)


def test_prefill_ignores_future_keys():
    rng = np.random.default_rng(10)
    N = 260
    Q, K, V = _rand(rng, 1, 2, N, 8), _rand(rng, 1, 1, N, 8), _rand(rng, 1, 1, N, 8)
    o = A.dense_prefill(Q, K, V)
    K2, V2 = K.copy(), V.copy()
    K2[0, 0, 200:] = 1e3
    V2[0, 0, 200:] = -7
    o2 = A.dense_prefill(Q, K2, V2)
    np.testing.assert_array_equal(o[:, :, :200], o2[:, :, :200])


def test_tile_weights_brute_force_and_sum():
    rng = np.random.default_rng(11)
    N, d = 200, 4
    Q, K = _rand(rng, 1, 1, N, d), _rand(rng, 1, 1, N, d)
    for t in range(A.n_tiles(N)):
        w = A.tile_weights(Q, K, 0, 0, t, [0], 0.7)
        r0, r1 = A.tile_rows(t, N)
        L = A.prefix_len(t, N)
        # pure-python loops: for every row, its own softmax over j <= i, summed per key
        wb = [0.0] * L
        for i in range(r0, r1):
            logits = [0.7 * sum(Q[0, 0, i, c] * K[0, 0, j, c] for c in range(d)) for j in range(i + 1)]
            mx = max(logits)
            ex = [math.exp(x - mx) for x in logits]
            z = sum(ex)
            for j in range(i + 1):
                wb[j] += ex[j] / z
        np.testing.assert_allclose(w, wb, atol=1e-12)
        np.testing.assert_allclose(w.sum(), r1 - r0, atol=1e-10)


def test_one_row_tile_weights_are_probabilities():
    rng = np.random.default_rng(12)
    N = 20
    Q, K = _rand(rng, 1, 1, N, 4), _rand(rng, 1, 1, N, 4)
    for t in range(N):
        w = A.tile_weights(Q, K, 0, 0, t, [0], 1.0, tile=1)
        p = A.softmax(K[0, 0, : t + 1] @ Q[0, 0, t])
        np.testing.assert_allclose(w, p, atol=1e-14)


def test_sparse_prefill_matches_masked_sdpa_and_empty_rows():
    rng = np.random.default_rng(13)
    B, Hq, Hkv, N, d, k = 1, 2, 1, 300, 8, 40
    Q, K, V = _rand(rng, B, Hq, N, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    nT = A.n_tiles(N)
    idx = np.full((B, Hq, nT, k), -1)
    mask = np.zeros((B, Hq, N, N), dtype=bool)
    for h in range(Hq):
        for t in range(nT):
            L = A.prefix_len(t, N)
            kt = min(k, L)
            sel = np.sort(rng.choice(np.arange(5, L), kt - 5, replace=False)) if L > 5 else np.zeros(0, int)
            idx[0, h, t, : sel.size] = sel
            r0, r1 = A.tile_rows(t, N)
            for i in range(r0, r1):
                mask[0, h, i, sel[sel <= i]] = True
    o = A.sparse_prefill(Q, K, V, idx)
    empty = ~mask.any(-1)
    assert empty.any()      # rows 0..4 see no selected key
    ref = _sdpa(Q, K[:, [0, 0]], V[:, [0, 0]], mask=mask | empty[..., None], scale=1 / math.sqrt(d))
    ref[empty] = 0.0
    np.testing.assert_allclose(o, ref, atol=1e-12)


def test_anchor_prefill_small_tiles_select_prefix_and_reuse_equals_dense():
    rng = np.random.default_rng(14)
    B, Hq, Hkv, N, d, k = 1, 2, 1, 384, 8, 256
    Q, K, V = _rand(rng, B, Hq, N, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    o_a, idx = A.anchor_prefill(Q, K, V, k)
    assert (idx[0, :, 0, :128] == np.arange(128)).all() and (idx[0, :, 0, 128:] == -1).all()
    assert (idx[0, :, 1, :256] == np.arange(256)).all()
    assert (idx[0, :, 2] >= 0).all() and (np.diff(idx[0, :, 2], axis=-1) > 0).all()
    o_r = A.sparse_prefill(Q, K, V, idx)
    np.testing.assert_allclose(o_r[:, :, :256], o_a[:, :, :256], atol=1e-12)
    # k >= N: every tile keeps its full prefix, reuse equals dense everywhere
    o_a2, idx2 = A.anchor_prefill(Q, K, V, N)
    np.testing.assert_allclose(A.sparse_prefill(Q, K, V, idx2), o_a2, atol=1e-12)


@pytest.mark.parametrize("gname", list(GMAPS))
def test_decode_unit_matches_sdpa_and_brute_force(gname):
    """decode_unit, the one-(sequence, head) form the full-size GPU checks use:
    its dense output equals the library routine on that head alone, its set
    is the brute-force Top-k of the head's logits under the tie rule (largest
    first, lower index on ties), and its sparse output equals the library
    routine with a mask holding only the given set."""
    rng = np.random.default_rng(31)
    B, Hq, Hkv, N, d, k = 2, 6, 2, 41, 8, 7
    gmap = GMAPS[gname]
    q, K, V = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    K[1, 0, 5] = K[1, 0, 9]                      # an exact logit tie inside the set
    for b, h in [(0, 0), (1, 3), (1, 4)]:
        g = gmap[h]
        o, idx, s = A.decode_unit(q, K, V, b, h, k, gmap, 0.4)
        ref = _sdpa(q[b, h][None, None, None], K[b, g][None, None], V[b, g][None, None],
                    scale=0.4)[0, 0, 0]
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
        # brute force: every key outside the set loses to every key inside it
        sel = set(idx.tolist())
        assert len(sel) == k and list(idx) == sorted(sel)
        for i in sel:
            for j in range(N):
                if j not in sel:
                    assert s[i] > s[j] or (s[i] == s[j] and i < j)
        # sparse form on an arbitrary set
        subset = np.sort(rng.choice(N, 9, replace=False))
        mask = np.zeros((1, 1, 1, N), dtype=bool)
        mask[..., subset] = True
        o_s = A.decode_unit(q, K, V, b, h, k, gmap, 0.4, idx=subset)
        ref_s = _sdpa(q[b, h][None, None, None], K[b, g][None, None], V[b, g][None, None],
                      mask=mask, scale=0.4)[0, 0, 0]
        np.testing.assert_allclose(o_s, ref_s, rtol=0, atol=1e-12)
