"""Layer-stack driver (oracle).

Anchor layers output exact attention and replace the held index sets;
reuse layers read the held sets unchanged, recomputing attention with their
own q, K, V (euno.news summary, Key Contributions "Cross-layer Top-k reuse",
Methodology 2-3). Layers before the first anchor have no sets to reuse and
run dense (the pages' example anchor list does not start at layer 0).
"""
from . import attention as A


def run_stack(mode, layers, k, anchors, group_map=None, scale=None, tile=A.TILE, pooled=False):
    """layers: list of (q, K, V) per layer. Returns (outputs, sets_read, sets_written).

    ``sets_read[l]`` is the index array layer l consumed (None for anchors and
    dense layers); anchors' own sets are returned in ``sets_written``. With
    ``pooled`` the sets are per (sequence, KV head) (GQA-pooled scores).
    """
    anchor_d = A.anchor_decode_pooled if pooled else A.anchor_decode
    sparse_d = A.sparse_decode_pooled if pooled else A.sparse_decode
    anchor_p = A.anchor_prefill_pooled if pooled else A.anchor_prefill
    sparse_p = A.sparse_prefill_pooled if pooled else A.sparse_prefill
    anchors = set(anchors)
    held = None
    outs, sets_read, sets_written = [], [], []
    for layer, (q, K, V) in enumerate(layers):
        if mode == "decode":
            if layer in anchors:
                o, held, _ = anchor_d(q, K, V, k, group_map, scale)
                sets_read.append(None)
                sets_written.append(held)
            elif held is None:
                o, _ = A.dense_decode(q, K, V, group_map, scale)
                sets_read.append(None)
                sets_written.append(None)
            else:
                o = sparse_d(q, K, V, held, group_map, scale)
                sets_read.append(held)
                sets_written.append(None)
        else:
            if layer in anchors:
                o, held = anchor_p(q, K, V, k, group_map, scale, tile)
                sets_read.append(None)
                sets_written.append(held)
            elif held is None:
                o = A.dense_prefill(q, K, V, group_map, scale, tile)
                sets_read.append(None)
                sets_written.append(None)
            else:
                o = sparse_p(q, K, V, held, group_map, scale, tile)
                sets_read.append(held)
                sets_written.append(None)
        outs.append(o)
    return outs, sets_read, sets_written
