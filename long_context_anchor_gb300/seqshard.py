"""Sequence-sharded (context-parallel) anchor decode across ranks.

The KV cache of every sequence is split along the key axis into one
contiguous shard per rank, in rank order (rank r holds the keys after those
of rank r - 1). Each rank runs ``kascade_anchor_decode_shard`` on its own
shard: the exact attention over the shard's keys, the shard's
log-normaliser and its local Top-k candidates (global positions and
logits). One exchange step, a single all-gather of those partials packed
into one byte buffer, gives every rank all of them, and
``kascade_merge_decode_shards`` turns them into the exact layer output and
the exact global Top-k: the union of the shards' local Top-k sets holds the
global one, so the same selection rule on the union finds it (the rule of
the Kascade anchor layer, euno.news summary, Methodology 2: exact attention,
then an exact per-head Top-k; the pages themselves run on one device).

This module holds the host side (packing, the collective, unpacking); the
arithmetic runs in the library's kernels.
"""
from typing import List, Sequence

import torch
import torch.distributed as dist


def _as_bytes(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(-1).view(torch.uint8)


def exchange_partials(tensors: Sequence[torch.Tensor], group=None) -> List[torch.Tensor]:
    """All-gather the given tensors over the group in one collective.

    The tensors are packed into one byte buffer per rank; the result holds,
    for each input tensor, a tensor of shape [world, *shape] whose entry r
    came from rank r. Every rank must pass tensors of the same shapes and
    dtypes in the same order."""
    world = dist.get_world_size(group)
    parts = [_as_bytes(t) for t in tensors]
    sizes = [p.numel() for p in parts]
    buf = torch.cat(parts)
    gathered = [torch.empty_like(buf) for _ in range(world)]
    dist.all_gather(gathered, buf, group=group)
    out = []
    off = 0
    for t, n in zip(tensors, sizes):
        rows = [g[off:off + n].view(t.dtype).view(t.shape) for g in gathered]
        out.append(torch.stack(rows))
        off += n
    return out


def sharded_anchor_decode(q, k_shard, v_shard, key_offset: int, topk: int, group=None,
                          group_map=None, scale=None, ws=None, stream=None):
    """Anchor decode layer over a cache sharded across the ranks of `group`.

    q [B,Hq,d] is the same on every rank; k_shard, v_shard [B,Hkv,N_r,d] are
    this rank's keys, which start at global position key_offset (ranks in
    key order; every shard holds at least topk keys). Returns (out [B,Hq,d],
    idx [B,Hq,topk] ascending global positions), the same on every rank."""
    from . import kascade as K
    part = K.anchor_decode_shard(q, k_shard, v_shard, key_offset, topk, group_map=group_map,
                                 scale=scale, ws=ws, stream=stream)
    outs, lses, cand_idx, cand_scores = exchange_partials(part, group)
    return K.merge_decode_shards(outs, lses, cand_idx, cand_scores, ws=ws, stream=stream)
