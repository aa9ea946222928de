"""Sequence-sharded anchor decode: per-shard partials and their exact merge (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages run Kascade on one device; they do not shard a sequence. This is
the context-parallel form of the anchor decode layer (euno.news summary,
Methodology 2: exact attention, then an exact per-head Top-k): the KV cache
of every sequence is split along the key axis into S contiguous shards, in
key order, and each shard produces

* o_s: exact attention of the query over the shard's keys only;
* lse_s = log sum_{j in shard} exp(s_j), the shard's log-normaliser;
* its local Top-k candidates (global positions, ascending) with their
  logits, under the library's one selection rule (larger logit first, lower
  position on ties).

One exchange step brings every shard's partials together, and the merge is
exact:

* output: with LSE = log sum_s exp(lse_s), o = sum_s exp(lse_s - LSE) o_s,
  which is the softmax over all keys written shard by shard;
* indices: every key of the global Top-k that lies in shard s is beaten by
  fewer than k keys overall, hence by fewer than k keys of shard s, so it is
  among shard s's own Top-k. The union of the shards' candidates therefore
  holds the global Top-k, and the same rule applied to the union (ties
  broken by global position) selects it exactly.

Each shard must hold at least k keys.
"""
import numpy as np

from .attention import dense_decode
from .topk import topk_indices


def logsumexp(s):
    """log sum exp over the last axis, with the maximum taken out first."""
    s = np.asarray(s, dtype=np.float64)
    m = s.max(axis=-1)
    return m + np.log(np.exp(s - m[..., None]).sum(axis=-1))


def decode_shard_partial(q, K_shard, V_shard, offset, k, group_map=None, scale=None):
    """One shard (global positions offset .. offset + N_s - 1) of every sequence.

    Returns (o_s [B,Hq,d], lse_s [B,Hq], cand_idx [B,Hq,k] int64 global
    positions ascending, cand_scores [B,Hq,k] the logits at those positions).
    """
    o, s = dense_decode(q, K_shard, V_shard, group_map, scale)
    B, Hq, n_s = s.shape
    if k > n_s:
        raise ValueError("a shard must hold at least k keys")
    lse = logsumexp(s)
    cand_idx = np.empty((B, Hq, k), dtype=np.int64)
    cand_scores = np.empty((B, Hq, k))
    for b in range(B):
        for h in range(Hq):
            local = topk_indices(s[b, h], k)
            cand_idx[b, h] = local + offset
            cand_scores[b, h] = s[b, h, local]
    return o, lse, cand_idx, cand_scores


def merge_decode_shards(parts, k):
    """parts: list over shards, in key order, of (o_s, lse_s, cand_idx, cand_scores).

    Returns (o [B,Hq,d], idx [B,Hq,k] ascending global positions).
    """
    lse = np.stack([p[1] for p in parts])                 # [S, B, Hq]
    m = lse.max(axis=0)
    wts = np.exp(lse - m[None])                          # exp(lse_s - max)
    o = sum(wts[s][..., None] * parts[s][0] for s in range(len(parts)))
    o = o / wts.sum(axis=0)[..., None]
    idx_all = np.concatenate([p[2] for p in parts], axis=-1)      # [B, Hq, S*k]
    sc_all = np.concatenate([p[3] for p in parts], axis=-1)
    B, Hq, _ = idx_all.shape
    idx = np.empty((B, Hq, k), dtype=np.int64)
    for b in range(B):
        for h in range(Hq):
            # score descending, then global position ascending
            order = np.lexsort((idx_all[b, h], -sc_all[b, h]))[:k]
            idx[b, h] = np.sort(idx_all[b, h][order])
    return o, idx


def shard_bounds(n, n_shards):
    """Contiguous key ranges [(offset, length)] splitting n keys into n_shards
    nearly equal shards (the first n % n_shards shards one key longer)."""
    base, extra = divmod(n, n_shards)
    out, off = [], 0
    for s in range(n_shards):
        ln = base + (1 if s < extra else 0)
        out.append((off, ln))
        off += ln
    return out


def sharded_anchor_decode(q, K, V, k, n_shards, group_map=None, scale=None):
    """The whole sharded layer: split K/V along the key axis, the shards'
    partials, then the merge. Returns (o, idx)."""
    parts = []
    for off, ln in shard_bounds(np.shape(K)[2], n_shards):
        parts.append(decode_shard_partial(q, np.asarray(K)[:, :, off:off + ln],
                                          np.asarray(V)[:, :, off:off + ln], off, k,
                                          group_map, scale))
    return merge_decode_shards(parts, k)

