"""Pins for oracle/shard.py (sequence-sharded anchor decode).

* The merged output equals torch's scaled_dot_product_attention in float64
  (a library routine) over the whole, unsharded cache, for uneven shards.
* The merged set equals the brute-force Top-k of the whole cache's logits:
  every selected key beats every unselected one (lower position on equal
  logits), including ties that straddle shard boundaries.
* Closed forms: with q = 0 every logit is 0, so each shard's log-normaliser
  is log(N_s) and its candidates are its first k positions.
* One shard is the unsharded anchor layer; the shard ranges tile the keys.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as A
from oracle import shard as S


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _sdpa_decode(q, K, V, gmap, scale):
    Kx, Vx = K[:, gmap], V[:, gmap]
    return F.scaled_dot_product_attention(torch.from_numpy(q[:, :, None, :]), torch.from_numpy(Kx),
                                          torch.from_numpy(Vx), scale=scale).numpy()[:, :, 0]


def _brute_force_ok(logits, sel):
    sel = set(int(i) for i in sel)
    for i in sel:
        for j in range(logits.shape[0]):
            if j not in sel:
                assert logits[i] > logits[j] or (logits[i] == logits[j] and i < j), (i, j)


@pytest.mark.parametrize("n_shards", [1, 2, 3, 5])
def test_merge_equals_unsharded_attention_and_topk(n_shards):
    rng = np.random.default_rng(40 + n_shards)
    B, Hq, Hkv, N, d, k = 2, 4, 2, 97, 8, 11
    gmap = [0, 0, 1, 1]
    q, K, V = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    o, idx = S.sharded_anchor_decode(q, K, V, k, n_shards, gmap, 0.35)
    np.testing.assert_allclose(o, _sdpa_decode(q, K, V, gmap, 0.35), rtol=0, atol=1e-12)
    s = A.decode_logits(q, K, gmap, 0.35)
    for b in range(B):
        for h in range(Hq):
            assert len(idx[b, h]) == k and (np.diff(idx[b, h]) > 0).all()
            _brute_force_ok(s[b, h], idx[b, h])


def test_ties_across_shard_boundaries():
    """Equal logits in different shards: the lower global position wins."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, N, d = 1, 2, 1, 40, 4
    q, K, V = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    big = 5.0 * q[0, 0] / np.linalg.norm(q[0, 0])
    # positions 3, 12, 25, 38 (one in each of four shards of 10) carry the same key
    for p in (3, 12, 25, 38):
        K[0, 0, p] = big
    gmap = [0, 0]
    for k in (1, 2, 3):
        o, idx = S.sharded_anchor_decode(q, K, V, k, 4, gmap, 1.0)
        # head 0: the four equal keys lead; the k lowest positions are taken
        assert idx[0, 0].tolist() == [3, 12, 25, 38][:k], (k, idx[0, 0])
        _, idx_ref, _ = A.anchor_decode(q, K, V, k, gmap, 1.0)
        assert np.array_equal(idx, idx_ref)


def test_zero_query_closed_form():
    rng = np.random.default_rng(3)
    B, Hq, Hkv, N, d, k = 1, 2, 2, 30, 4, 5
    q = np.zeros((B, Hq, d))
    K, V = _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    for off, ln in S.shard_bounds(N, 3):
        o, lse, ci, cs = S.decode_shard_partial(q, K[:, :, off:off + ln], V[:, :, off:off + ln],
                                                off, k)
        np.testing.assert_allclose(lse, math.log(ln), rtol=0, atol=1e-14)
        assert (ci == np.arange(off, off + k)).all() and (cs == 0.0).all()
        np.testing.assert_allclose(o, V[:, :, off:off + ln].mean(axis=2), atol=1e-14)


def test_one_shard_is_the_anchor_layer_and_bounds_tile():
    rng = np.random.default_rng(5)
    q, K, V = _rand(rng, 1, 4, 8), _rand(rng, 1, 2, 50, 8), _rand(rng, 1, 2, 50, 8)
    o, idx = S.sharded_anchor_decode(q, K, V, 9, 1)
    o_ref, idx_ref, _ = A.anchor_decode(q, K, V, 9)
    np.testing.assert_array_equal(idx, idx_ref)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-15)
    for n, s in [(50, 1), (50, 3), (7, 7), (1000, 6)]:
        b = S.shard_bounds(n, s)
        assert b[0][0] == 0 and sum(ln for _, ln in b) == n
        assert all(b[i][0] + b[i][1] == b[i + 1][0] for i in range(s - 1))
        assert max(ln for _, ln in b) - min(ln for _, ln in b) <= 1
    with pytest.raises(ValueError):
        S.decode_shard_partial(q, K[:, :, :5], V[:, :, :5], 0, 9)
