"""GPU parity of the sequence-sharded anchor decode, through the C ABI, with
the shards run one after another on the one GPU: every shard's partials
(kascade_anchor_decode_shard), then the merge (kascade_merge_decode_shards).
The merged index sets must equal the unsharded anchor layer's bit for bit
(the shards rank the same fp32 logits), and the Top-k rule of the oracle on
those logits; the merged output must match the float64 oracle; each shard's
log-normaliser matches the oracle's. The exchange step is then run for real
on a one-rank NCCL group."""
import os
import socket

import numpy as np
import pytest
import torch

import __graft_entry__
from gpu_helpers import check_index_set, check_out, check_topk_exact, f64
from oracle import attention as A
from oracle import shard as S

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def K():
    __graft_entry__.build()
    from long_context_anchor_gb300 import kascade
    return kascade


def _layer(B, Hq, Hkv, N, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, d, generator=g)
    k = torch.randn(B, Hkv, N, d, generator=g)
    v = torch.randn(B, Hkv, N, d, generator=g)
    return [x.to(dtype).to(DEV) for x in (q, k, v)]


def _shards(K, q, k, v, topk, n_shards):
    parts = []
    for off, ln in S.shard_bounds(k.shape[2], n_shards):
        ks, vs = k[:, :, off:off + ln].contiguous(), v[:, :, off:off + ln].contiguous()
        parts.append((off, ln) + K.anchor_decode_shard(q, ks, vs, off, topk))
    return parts


CASES = [  # B, Hq, Hkv, N, d, dtype, topk, shards
    (2, 32, 8, 32768, 128, torch.bfloat16, 4096, 2),
    (2, 32, 8, 32768, 128, torch.bfloat16, 4096, 4),
    (1, 64, 8, 131072, 64, torch.bfloat16, 8192, 8),
    (1, 8, 2, 3001, 64, torch.bfloat16, 300, 3),      # uneven shards
    (1, 4, 2, 999, 64, torch.float32, 50, 5),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_sharded_anchor_decode_matches_unsharded_and_oracle(K, case):
    B, Hq, Hkv, N, d, dtype, topk, n_shards = CASES[case]
    q, k, v = _layer(B, Hq, Hkv, N, d, dtype, seed=100 + case)
    out_u, idx_u, s_u = K.anchor_decode(q, k, v, topk, return_scores=True)
    parts = _shards(K, q, k, v, topk, n_shards)
    s_np = s_u.cpu().numpy()
    Q, Kh, V = f64(q), f64(k), f64(v)
    for off, ln, o_s, lse_s, ci, cs in parts:
        ci_np = ci.cpu().numpy()
        # the shard ranked the very logits the unsharded layer ranks
        got = np.take_along_axis(s_np, ci_np.astype(np.int64), axis=2)
        assert np.array_equal(cs.cpu().numpy(), got), (off, "candidate logits differ")
        assert (ci_np >= off).all() and (ci_np < off + ln).all()
        # the shard's log-normaliser and output against the oracle's partial
        o_ref, lse_ref, _, _ = S.decode_shard_partial(Q, Kh[:, :, off:off + ln],
                                                      V[:, :, off:off + ln], off, topk)
        tol = 1e-4 if dtype == torch.float32 else 1e-3
        assert np.abs(lse_s.cpu().numpy() - lse_ref).max() < tol
        if dtype == torch.float32:
            check_out(o_s, o_ref, 1e-4, 1e-5)
        else:
            check_out(o_s, o_ref)
    stack = lambda i: torch.stack([p[i] for p in parts])
    out_m, idx_m = K.merge_decode_shards(stack(2), stack(3), stack(4), stack(5), kv_len=N)
    torch.cuda.synchronize()
    # bit-exact: the merge selects the unsharded layer's sets
    assert torch.equal(idx_m, idx_u)
    o_ref, _, s_ref = A.anchor_decode(Q, Kh, V, topk)
    if dtype == torch.float32:
        check_out(out_m, o_ref, 1e-4, 1e-5)
    else:
        check_out(out_m, o_ref)
    got = idx_m.cpu().numpy()
    rng = np.random.default_rng(case)
    for b, h in [(0, 0), (B - 1, Hq - 1), (int(rng.integers(B)), int(rng.integers(Hq)))]:
        check_topk_exact(got[b, h], s_np[b, h], topk, what=("merged top-k", b, h))
        check_index_set(got[b, h], s_ref[b, h], topk, what=("merged set", b, h))


def test_merge_reports_shards_out_of_order(K):
    q, k, v = _layer(1, 8, 2, 2048, 128, torch.bfloat16, seed=9)
    parts = _shards(K, q, k, v, 64, 2)[::-1]          # key order reversed
    stack = lambda i: torch.stack([p[i] for p in parts])
    ws = K.Workspace(DEV)
    K.merge_decode_shards(stack(2), stack(3), stack(4), stack(5), kv_len=2048, ws=ws)
    assert ws.device_error() == K.BAD_INPUT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_exchange_over_nccl_one_rank(K):
    """The product path of the multi-device form (local partials, the one
    all-gather, the merge) on a one-rank NCCL group: it equals the unsharded
    anchor layer."""
    import torch.distributed as dist
    from long_context_anchor_gb300.seqshard import sharded_anchor_decode
    q, k, v = _layer(2, 16, 4, 8192, 128, torch.bfloat16, seed=5)
    out_u, idx_u = K.anchor_decode(q, k, v, 1024)
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    os.environ["NCCL_NVLS_ENABLE"] = "0"        # plain transport only
    dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % _free_port(), rank=0,
                            world_size=1, device_id=DEV)
    try:
        out, idx = sharded_anchor_decode(q, k, v, 0, 1024)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert torch.equal(idx, idx_u)
    check_out(out, A.dense_decode(f64(q), f64(k), f64(v))[0])
