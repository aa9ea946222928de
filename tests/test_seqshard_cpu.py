"""The exchange step of the sequence-sharded anchor decode on CPU: world_size-2
gloo ranks (rendezvous on 127.0.0.1), each holding one contiguous shard of
the keys. Each rank computes its partials with the oracle, the library's
host-side exchange (one all-gather of the packed partials) brings both
shards' partials to every rank in rank order, and the oracle's merge of
what arrived equals the unsharded oracle: the same output, and the same
index sets bit for bit, ties across the shard boundary included."""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    rng = np.random.default_rng(77)
    B, Hq, Hkv, N, d = 2, 4, 2, 300, 16
    q = rng.standard_normal((B, Hq, d))
    K = rng.standard_normal((B, Hkv, N, d))
    V = rng.standard_normal((B, Hkv, N, d))
    # equal keys on both sides of the boundary (positions 140 and 160)
    K[0, 0, 160] = K[0, 0, 140] = 4.0 * q[0, 0] / np.linalg.norm(q[0, 0])
    return q, K, V


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from long_context_anchor_gb300.seqshard import exchange_partials
        from oracle import shard as S
        q, K, V = _inputs()
        k = 37
        off, ln = S.shard_bounds(K.shape[2], world)[rank]
        o, lse, ci, cs = S.decode_shard_partial(q, K[:, :, off:off + ln], V[:, :, off:off + ln],
                                                off, k)
        mine = [torch.from_numpy(x) for x in (o, lse, ci.astype(np.int32), cs.astype(np.float32))]
        got = exchange_partials(mine, None)
        # rank order = shard order; this rank's own entry came back unchanged
        assert [g.shape[0] for g in got] == [world] * 4
        for g, m in zip(got, mine):
            assert torch.equal(g[rank], m)
        parts = [tuple(g[s].numpy() for g in got) for s in range(world)]
        o_m, idx_m = S.merge_decode_shards(parts, k)
        out[rank] = (o_m, idx_m)
    finally:
        dist.destroy_process_group()


def test_exchange_then_merge_equals_unsharded_world2():
    from oracle import attention as A
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:   # no fork of a threaded process
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    q, K, V = _inputs()
    o_ref, idx_ref, _ = A.anchor_decode(q, K, V, 37)
    for r in range(world):
        o_m, idx_m = res[r]
        np.testing.assert_array_equal(idx_m, idx_ref)
        np.testing.assert_allclose(o_m, o_ref, rtol=0, atol=1e-12)
    # the tie straddles the boundary; the lower position leads the set
    assert 140 in idx_ref[0, 0] and 160 in idx_ref[0, 0]
