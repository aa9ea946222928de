"""Dense, anchor and reuse attention in float64 (oracle).

Notation (Kascade pages; shapes are the library's):

* decode: q [B, Hq, d], K, V [B, Hkv, N, d]; one query per sequence sees all
  N cached keys (no mask);
* prefill: Q [B, Hq, N, d], K, V [B, Hkv, N, d]; row i sees keys j <= i;
* g(h) = group_map[h] is the KV head query head h reads (GQA);
* scale sigma defaults to 1/sqrt(d) (the pages give no scale; this is the
  standard attention scale).

Anchor layers compute attention exactly and take an exact Top-k per head
(euno.news summary, Methodology 2 and 5). Reuse layers recompute the logits
with their own q, K, V but restrict the softmax to the saved index set
(Methodology 3). Prefill uses one index set per (head, query tile of 128
rows) (opentrain.ai Abstract, "tile-level operations"), ranked by the tile's
summed post-softmax weights and capped at the tile's causal prefix.
"""
import math

import numpy as np

from .topk import topk_indices

TILE = 128


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def default_group_map(n_q_heads: int, n_kv_heads: int):
    g = n_q_heads // n_kv_heads
    return [h // g for h in range(n_q_heads)]


def softmax(s):
    """Row softmax over the last axis: exp(s - max) / sum exp(s - max)."""
    s = _f64(s)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


# ----------------------------------------------------------------- decode --

def decode_logits(q, K, group_map, scale):
    """s[b, h, j] = sigma * q[b, h] . K[b, g(h), j]   -> [B, Hq, N] float64."""
    q, K = _f64(q), _f64(K)
    B, Hq, _ = q.shape
    s = np.empty((B, Hq, K.shape[2]))
    for b in range(B):
        for h in range(Hq):
            s[b, h] = scale * (K[b, group_map[h]] @ q[b, h])
    return s


def dense_decode(q, K, V, group_map=None, scale=None):
    """Exact attention for one query per sequence. Returns (o [B,Hq,d], s [B,Hq,N])."""
    B, Hq, d = np.shape(q)
    group_map = group_map if group_map is not None else default_group_map(Hq, np.shape(K)[1])
    scale = default_scale(d) if scale is None else scale
    s = decode_logits(q, K, group_map, scale)
    p = softmax(s)
    V = _f64(V)
    o = np.empty((B, Hq, d))
    for b in range(B):
        for h in range(Hq):
            o[b, h] = p[b, h] @ V[b, group_map[h]]
    return o, s


def anchor_decode(q, K, V, k, group_map=None, scale=None):
    """Anchor layer: exact output plus the per-(sequence, head) Top-k of the logits.

    Ranking by logits selects the same set as ranking by softmax weights
    (softmax is monotone within a row) without ties created by exp underflow.
    Returns (o, idx [B, Hq, min(k, N)] ascending int64, s).
    """
    o, s = dense_decode(q, K, V, group_map, scale)
    B, Hq, N = s.shape
    kk = min(k, N)
    idx = np.empty((B, Hq, kk), dtype=np.int64)
    for b in range(B):
        for h in range(Hq):
            idx[b, h] = topk_indices(s[b, h], kk)
    return o, idx, s


def sparse_decode(q, K, V, idx, group_map=None, scale=None):
    """Reuse layer: softmax restricted to the saved set S = idx[b, h].

    o = sum_{j in S} softmax_S(sigma q . K_j) V_j, with this layer's q, K, V.
    Rows of K and V outside S are never read.
    """
    B, Hq, d = np.shape(q)
    group_map = group_map if group_map is not None else default_group_map(Hq, np.shape(K)[1])
    scale = default_scale(d) if scale is None else scale
    q = _f64(q)
    o = np.empty((B, Hq, d))
    for b in range(B):
        for h in range(Hq):
            sel = np.asarray(idx[b, h], dtype=np.int64)
            Ks = _f64(K[b, group_map[h]][sel])
            Vs = _f64(V[b, group_map[h]][sel])
            p = softmax(scale * (Ks @ q[b, h]))
            o[b, h] = p @ Vs
    return o


def decode_unit(q, K, V, b, h, k, group_map, scale, idx=None):
    """One (sequence, head) unit, for sampled checks at full size.

    Dense/anchor when ``idx`` is None (returns o, idx, s), sparse otherwise
    (returns o).
    """
    g = group_map[h]
    qv = _f64(q[b, h])
    if idx is None:
        s = scale * (_f64(K[b, g]) @ qv)
        o = softmax(s) @ _f64(V[b, g])
        return o, topk_indices(s, k), s
    sel = np.asarray(idx, dtype=np.int64)
    p = softmax(scale * (_f64(K[b, g][sel]) @ qv))
    return p @ _f64(V[b, g][sel])


# ---------------------------------------------------------------- prefill --

def n_tiles(n: int, tile: int = TILE) -> int:
    return (n + tile - 1) // tile


def tile_rows(t: int, n: int, tile: int = TILE):
    return t * tile, min(n, (t + 1) * tile)


def prefix_len(t: int, n: int, tile: int = TILE) -> int:
    """L_t: number of keys the last row of tile t can see."""
    return min(n, (t + 1) * tile)


def prefill_tile_logits(Q, K, b, h, t, group_map, scale, tile=TILE):
    """sigma * Q[b,h,i] . K[b,g(h),j] for rows i of tile t and j < L_t; -inf where j > i."""
    n = np.shape(Q)[2]
    r0, r1 = tile_rows(t, n, tile)
    L = prefix_len(t, n, tile)
    s = scale * (_f64(Q[b, h, r0:r1]) @ _f64(K[b, group_map[h], :L]).T)
    rows = np.arange(r0, r1)[:, None]
    cols = np.arange(L)[None, :]
    s[cols > rows] = -np.inf
    return s


def dense_prefill_tile(Q, K, V, b, h, t, group_map, scale, tile=TILE):
    """Causal exact attention for the rows of one tile. Returns (o [rows, d], lse [rows])."""
    s = prefill_tile_logits(Q, K, b, h, t, group_map, scale, tile)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=1, keepdims=True)
    L = s.shape[1]
    o = (e / z) @ _f64(V[b, group_map[h], :L])
    lse = (m + np.log(z))[:, 0]
    return o, lse


def tile_weights(Q, K, b, h, t, group_map, scale, tile=TILE):
    """w_j = sum over the tile's rows i (i >= j) of the post-softmax weight p_ij, j < L_t."""
    s = prefill_tile_logits(Q, K, b, h, t, group_map, scale, tile)
    return softmax(s).sum(axis=0)


def anchor_prefill_tile(Q, K, V, b, h, t, k, group_map, scale, tile=TILE):
    """Anchor layer, one (head, tile): exact rows, tile weights, Top-k_t of the weights.

    k_t = min(k, L_t): the set is capped at the causal prefix of the tile.
    Returns (o, idx ascending, w).
    """
    o, _ = dense_prefill_tile(Q, K, V, b, h, t, group_map, scale, tile)
    w = tile_weights(Q, K, b, h, t, group_map, scale, tile)
    kt = min(k, w.shape[0])
    return o, topk_indices(w, kt), w


def sparse_prefill_tile(Q, K, V, idx, b, h, t, group_map, scale, tile=TILE):
    """Reuse layer, one (head, tile): row i attends to S_i = {j in S_t : j <= i}.

    ``idx`` is the tile's saved set (entries < 0 are padding and ignored).
    A row whose S_i is empty outputs zeros.
    Returns (o [rows, d], lse [rows]) with lse = -inf for empty rows.
    """
    n = np.shape(Q)[2]
    r0, r1 = tile_rows(t, n, tile)
    sel = np.asarray(idx, dtype=np.int64)
    sel = sel[sel >= 0]
    g = group_map[h]
    d = np.shape(Q)[3]
    o = np.zeros((r1 - r0, d))
    lse = np.full(r1 - r0, -np.inf)
    if sel.size == 0:
        return o, lse
    s = scale * (_f64(Q[b, h, r0:r1]) @ _f64(K[b, g][sel]).T)
    rows = np.arange(r0, r1)[:, None]
    s[sel[None, :] > rows] = -np.inf
    Vs = _f64(V[b, g][sel])
    for r in range(r1 - r0):
        if np.isneginf(s[r]).all():
            continue
        m = s[r].max()
        e = np.exp(s[r] - m)
        z = e.sum()
        o[r] = (e / z) @ Vs
        lse[r] = m + math.log(z)
    return o, lse


def dense_prefill(Q, K, V, group_map=None, scale=None, tile=TILE):
    """Whole-sequence causal attention, tile by tile. Returns o [B, Hq, N, d]."""
    B, Hq, N, d = np.shape(Q)
    group_map = group_map if group_map is not None else default_group_map(Hq, np.shape(K)[1])
    scale = default_scale(d) if scale is None else scale
    o = np.empty((B, Hq, N, d))
    for b in range(B):
        for h in range(Hq):
            for t in range(n_tiles(N, tile)):
                r0, r1 = tile_rows(t, N, tile)
                o[b, h, r0:r1] = dense_prefill_tile(Q, K, V, b, h, t, group_map, scale, tile)[0]
    return o


def anchor_prefill(Q, K, V, k, group_map=None, scale=None, tile=TILE):
    """Anchor layer over the whole sequence.

    Returns (o [B,Hq,N,d], idx [B,Hq,nT,k] int64 ascending, padded with -1
    beyond k_t = min(k, L_t)).
    """
    B, Hq, N, d = np.shape(Q)
    group_map = group_map if group_map is not None else default_group_map(Hq, np.shape(K)[1])
    scale = default_scale(d) if scale is None else scale
    nT = n_tiles(N, tile)
    o = np.empty((B, Hq, N, d))
    idx = np.full((B, Hq, nT, k), -1, dtype=np.int64)
    for b in range(B):
        for h in range(Hq):
            for t in range(nT):
                r0, r1 = tile_rows(t, N, tile)
                ot, it, _ = anchor_prefill_tile(Q, K, V, b, h, t, k, group_map, scale, tile)
                o[b, h, r0:r1] = ot
                idx[b, h, t, :it.shape[0]] = it
    return o, idx


def sparse_prefill(Q, K, V, idx, group_map=None, scale=None, tile=TILE):
    """Reuse layer over the whole sequence with saved sets idx [B,Hq,nT,k]."""
    B, Hq, N, d = np.shape(Q)
    group_map = group_map if group_map is not None else default_group_map(Hq, np.shape(K)[1])
    scale = default_scale(d) if scale is None else scale
    o = np.empty((B, Hq, N, d))
    for b in range(B):
        for h in range(Hq):
            for t in range(n_tiles(N, tile)):
                r0, r1 = tile_rows(t, N, tile)
                o[b, h, r0:r1] = sparse_prefill_tile(Q, K, V, idx[b, h, t], b, h, t,
                                                     group_map, scale, tile)[0]
    return o


# ---------------------------------------------------- GQA-pooled index sets --
#
# One index set per (sequence, KV head) instead of per query head. The pages
# give each attention head its own Top-k list (euno.news summary,
# Methodology 5) and run GQA models (Llama-3.1-8B: 32 query heads over 8 KV
# heads); they leave open how a group's heads would share one list. The
# reading taken here: the score of key j for KV head g is the sum over the
# group's query heads h (g(h) = g) of their post-softmax weights p_hj in
# decode, and of the tile weights w_{t,h,j} in prefill. The selection rule is
# unchanged; every query head of a group then attends over the group's set.

def pooled_decode_weights(s, group_map, n_kv_heads):
    """w[b, g, j] = sum over heads h with g(h) = g of softmax(s[b, h])_j -> [B, Hkv, N]."""
    p = softmax(s)
    B, Hq, N = p.shape
    w = np.zeros((B, n_kv_heads, N))
    for h in range(Hq):
        w[:, group_map[h]] += p[:, h]
    return w


def anchor_decode_pooled(q, K, V, k, group_map=None, scale=None):
    """Anchor layer with one set per (sequence, KV head).

    Returns (o [B,Hq,d], idx [B,Hkv,min(k,N)] ascending int64, w [B,Hkv,N]).
    """
    B, Hq, _ = np.shape(q)
    Hkv = np.shape(K)[1]
    group_map = group_map if group_map is not None else default_group_map(Hq, Hkv)
    o, s = dense_decode(q, K, V, group_map, scale)
    w = pooled_decode_weights(s, group_map, Hkv)
    kk = min(k, w.shape[2])
    idx = np.empty((B, Hkv, kk), dtype=np.int64)
    for b in range(B):
        for g in range(Hkv):
            idx[b, g] = topk_indices(w[b, g], kk)
    return o, idx, w


def expand_pooled_sets(idx, group_map):
    """Per-query-head view of per-KV-head sets: out[:, h] = idx[:, g(h)]."""
    return np.asarray(idx)[:, list(group_map)]


def sparse_decode_pooled(q, K, V, idx, group_map=None, scale=None):
    """Reuse layer over per-KV-head sets idx [B,Hkv,k]: head h attends over S_{g(h)}."""
    Hq, Hkv = np.shape(q)[1], np.shape(K)[1]
    group_map = group_map if group_map is not None else default_group_map(Hq, Hkv)
    return sparse_decode(q, K, V, expand_pooled_sets(idx, group_map), group_map, scale)


def tile_weights_pooled(Q, K, b, g, t, group_map, scale, tile=TILE):
    """sum over heads h with g(h) = g of the tile weights w_{t,h,j}, j < L_t."""
    heads = [h for h in range(len(group_map)) if group_map[h] == g]
    w = None
    for h in heads:
        wh = tile_weights(Q, K, b, h, t, group_map, scale, tile)
        w = wh if w is None else w + wh
    return w


def anchor_prefill_pooled(Q, K, V, k, group_map=None, scale=None, tile=TILE):
    """Anchor layer, prefill, one set per (sequence, KV head, tile).

    Returns (o [B,Hq,N,d], idx [B,Hkv,nT,k] int64 ascending, -1 padded
    beyond k_t = min(k, L_t)).
    """
    B, Hq, N, d = np.shape(Q)
    Hkv = np.shape(K)[1]
    group_map = group_map if group_map is not None else default_group_map(Hq, Hkv)
    scale = default_scale(d) if scale is None else scale
    o = dense_prefill(Q, K, V, group_map, scale, tile)
    nT = n_tiles(N, tile)
    idx = np.full((B, Hkv, nT, k), -1, dtype=np.int64)
    for b in range(B):
        for g in range(Hkv):
            for t in range(nT):
                w = tile_weights_pooled(Q, K, b, g, t, group_map, scale, tile)
                it = topk_indices(w, min(k, w.shape[0]))
                idx[b, g, t, :it.shape[0]] = it
    return o, idx


def sparse_prefill_pooled(Q, K, V, idx, group_map=None, scale=None, tile=TILE):
    """Reuse layer, prefill, over per-KV-head tile sets idx [B,Hkv,nT,k]."""
    Hq, Hkv = np.shape(Q)[1], np.shape(K)[1]
    group_map = group_map if group_map is not None else default_group_map(Hq, Hkv)
    return sparse_prefill(Q, K, V, expand_pooled_sets(idx, group_map), group_map, scale, tile)
