"""GPU parity of the tiled causal prefill path (tcgen05 kernels) against the
float64 oracle, through the C ABI: dense prefill, anchor prefill (exact rows
plus per-(head, 128-row tile) Top-k of the summed post-softmax weights) and
reuse prefill over saved tile sets."""
import numpy as np
import pytest
import torch

import __graft_entry__
from long_context_anchor_gb300 import configs
from long_context_anchor_gb300.workloads import make_layers, group_map as default_gmap
from oracle import attention as A
from oracle.stack import run_stack as run_oracle_stack
from oracle.topk import topk_indices
from gpu_helpers import (check_index_set, check_out, check_topk_exact, check_weights, f64,
                         log_w, packed_tile)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def K():
    __graft_entry__.build()
    from long_context_anchor_gb300 import kascade
    return kascade


def _dev_idx(idx):
    """Oracle index sets as the int32 device tensor the library takes."""
    return torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to(DEV)


def _layer(B, Hq, Hkv, N, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, N, d, generator=g)
    k = torch.randn(B, Hkv, N, d, generator=g)
    v = torch.randn(B, Hkv, N, d, generator=g)
    return [x.to(torch.bfloat16).to(DEV) for x in (q, k, v)]


SHAPES = [  # B, Hq, Hkv, N
    (1, 2, 1, 128),       # one tile
    (1, 4, 2, 300),       # ragged last tile
    (2, 8, 2, 520),       # G = 4, batch 2, ragged
    (1, 8, 1, 1024),      # G = 8
]


@pytest.mark.parametrize("shape", SHAPES)
def test_dense_prefill_matches_oracle(K, shape):
    B, Hq, Hkv, N = shape
    q, k, v = _layer(B, Hq, Hkv, N, 128, seed=N + Hq)
    out = K.dense_prefill(q, k, v)
    ref = A.dense_prefill(f64(q), f64(k), f64(v))
    check_out(out, ref)


def test_dense_prefill_permuted_map_and_scale(K):
    gm = [1, 0, 0, 1]
    q, k, v = _layer(1, 4, 2, 260, 128, seed=3)
    out = K.dense_prefill(q, k, v, group_map=gm, scale=0.05)
    check_out(out, A.dense_prefill(f64(q), f64(k), f64(v), gm, 0.05))


@pytest.mark.parametrize("shape,topk", [((1, 4, 2, 300), 64), ((2, 8, 2, 520), 130),
                                        ((1, 8, 1, 1024), 128), ((1, 2, 1, 1000), 1000)])
def test_anchor_prefill_matches_oracle(K, shape, topk):
    """Every (sequence, head, tile): the kernel's tile weights against the
    oracle's element by element, its packed-row Top-k bit-exact against the
    oracle rule on those identical fp32 weights, and its set against the
    oracle's own float64 set (near-ties judged on log-weights)."""
    B, Hq, Hkv, N = shape
    q, k, v = _layer(B, Hq, Hkv, N, 128, seed=5 * N + topk)
    out, idx, wts = K.anchor_prefill(q, k, v, topk, return_weights=True)
    assert wts.shape == (B, Hq, K.packed_tile_len(N))
    Q, Kh, V = f64(q), f64(k), f64(v)
    gm = A.default_group_map(Hq, Hkv)
    scale = 1.0 / np.sqrt(128)
    check_out(out, A.dense_prefill(Q, Kh, V))
    got = idx.cpu().numpy()
    w_gpu = wts.cpu().numpy()
    nT = A.n_tiles(N)
    for b in range(B):
        for h in range(Hq):
            for t in range(nT):
                w_ref = A.tile_weights(Q, Kh, b, h, t, gm, scale)
                w_row = packed_tile(w_gpu[b, h], t, N)
                check_weights(w_row, w_ref, what=("tile weights", b, h, t))
                kt = min(topk, w_ref.shape[0])
                row = got[b, h, t]
                check_topk_exact(row, w_row, kt, what=("tile top-k", b, h, t))
                check_index_set(row[:kt], log_w(w_ref), kt, what=("tile set", b, h, t))
    # the weights buffer is optional: without it the sets are the same
    _, idx2 = K.anchor_prefill(q, k, v, topk)
    assert torch.equal(idx, idx2)


@pytest.mark.parametrize("shape,topk", [((1, 4, 2, 300), 64), ((2, 8, 2, 520), 130)])
def test_reuse_prefill_matches_oracle(K, shape, topk):
    B, Hq, Hkv, N = shape
    q, k, v = _layer(B, Hq, Hkv, N, 128, seed=7 * N)
    _, idx_ref = A.anchor_prefill(f64(q), f64(k), f64(v), topk)   # the oracle's tile sets
    q2, k2, v2 = _layer(B, Hq, Hkv, N, 128, seed=9 * N)
    out = K.reuse_prefill(q2, k2, v2, _dev_idx(idx_ref))
    check_out(out, A.sparse_prefill(f64(q2), f64(k2), f64(v2), idx_ref))


def test_reuse_prefill_empty_rows_and_all_keys(K):
    B, Hq, Hkv, N, topk = 1, 2, 1, 384, 40
    q, k, v = _layer(B, Hq, Hkv, N, 128, seed=11)
    nT = A.n_tiles(N)
    rng = np.random.default_rng(0)
    idx = np.full((B, Hq, nT, topk), -1, dtype=np.int32)
    for h in range(Hq):
        for t in range(nT):
            L = min(N, 128 * (t + 1))
            # no saved key below position 20: rows 0..19 see an empty set
            sel = np.sort(rng.choice(np.arange(20, L), min(topk, L - 20), replace=False))
            idx[0, h, t, :sel.size] = sel
    idx_t = torch.from_numpy(idx).to(DEV)
    out = K.reuse_prefill(q, k, v, idx_t)
    ref = A.sparse_prefill(f64(q), f64(k), f64(v), idx)
    check_out(out, ref)
    assert float(out[0, :, :20].float().abs().max()) == 0.0
    # k >= N: every tile keeps its whole causal prefix -> reuse equals dense
    _, idx_all = K.anchor_prefill(q, k, v, N)
    out_r = K.reuse_prefill(q, k, v, idx_all)
    out_d = K.dense_prefill(q, k, v)
    assert (out_r.float() - out_d.float()).abs().max().item() < 1e-2


def test_reuse_prefill_poison_unselected_rows(K):
    B, Hq, Hkv, N, topk = 1, 4, 2, 512, 96
    q, k, v = _layer(B, Hq, Hkv, N, 128, seed=13)
    _, idx = K.anchor_prefill(q, k, v, topk)
    out = K.reuse_prefill(q, k, v, idx)
    used = torch.zeros(B, Hkv, N, dtype=torch.bool, device=DEV)
    gm = default_gmap(Hq, Hkv)
    for h in range(Hq):
        sel = idx[0, h].reshape(-1)
        sel = sel[sel >= 0].long()
        used[0, gm[h], sel] = True
    kp, vp = k.clone(), v.clone()
    kp[~used] = float("nan")
    vp[~used] = float("nan")
    assert torch.equal(K.reuse_prefill(q, kp, vp, idx), out)


def test_prefill_stack_matches_layer_calls(K):
    w = configs.LLAMA8B_PREFILL_16K.with_(n_layers=4, kv_len=640, topk=80, anchors=(1,))
    qs, ks, vs = make_layers(w, device=DEV)
    outs, idx_buf = K.run_stack(K.PREFILL, qs, ks, vs, w.topk, [1])
    o0 = K.dense_prefill(qs[0], ks[0], vs[0])
    o1, i1 = K.anchor_prefill(qs[1], ks[1], vs[1], w.topk)
    o2 = K.reuse_prefill(qs[2], ks[2], vs[2], i1)
    o3 = K.reuse_prefill(qs[3], ks[3], vs[3], i1)
    for a_, b_ in zip(outs, [o0, o1, o2, o3]):
        assert torch.equal(a_, b_)
    assert torch.equal(idx_buf, i1)
    # against the oracle stack, which selects its own float64 tile sets
    ref_outs, _, _ = run_oracle_stack("prefill", [(f64(a_), f64(b_), f64(c_))
                                                  for a_, b_, c_ in zip(qs, ks, vs)], w.topk, [1])
    for o, r in zip(outs, ref_outs):
        check_out(o, r)


def test_full_size_prefill_sampled(K):
    """The Llama-3.1-8B prefill shape at N = 16384 (k = 2048) through the stack
    call, on sampled (head, tile) units including the first and last tiles:
    anchor rows, tile weights, the bit-exact packed-row Top-k and the tile set
    against the oracle, and the reuse rows over the oracle's own set."""
    w = configs.LLAMA8B_PREFILL_16K.with_(n_layers=2)
    qs, ks, vs = make_layers(w, device=DEV)
    outs, idx = K.run_stack(K.PREFILL, qs, ks, vs, w.topk, [0])
    # the anchor entry point with the weights buffer gives the stack's sets
    _, idx_a, wts = K.anchor_prefill(qs[0], ks[0], vs[0], w.topk, return_weights=True)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_a)
    gm = default_gmap(w.n_q_heads, w.n_kv_heads)
    scale = 1.0 / np.sqrt(w.head_dim)
    nT = A.n_tiles(w.kv_len)
    rng = np.random.default_rng(2)
    units = [(0, 0), (w.n_q_heads - 1, nT - 1), (5, 20)] + \
        [(int(rng.integers(w.n_q_heads)), int(rng.integers(nT))) for _ in range(3)]
    idx_np = idx.cpu().numpy()
    # host copies of the sampled heads' rows only
    Q0, Q1 = f64(qs[0]), f64(qs[1])
    K0, V0, K1, V1 = f64(ks[0]), f64(vs[0]), f64(ks[1]), f64(vs[1])
    for h, t in units:
        r0, r1 = A.tile_rows(t, w.kv_len)
        o_ref, _ = A.dense_prefill_tile(Q0, K0, V0, 0, h, t, gm, scale)
        check_out(outs[0][0, h, r0:r1], o_ref, what=("anchor rows", h, t))
        w_ref = A.tile_weights(Q0, K0, 0, h, t, gm, scale)
        w_row = packed_tile(wts[0, h].cpu().numpy(), t, w.kv_len)
        check_weights(w_row, w_ref, what=("tile weights", h, t))
        kt = min(w.topk, w_ref.shape[0])
        check_topk_exact(idx_np[0, h, t], w_row, kt, what=("tile top-k", h, t))
        check_index_set(idx_np[0, h, t, :kt], log_w(w_ref), kt, what=("tile set", h, t))
        sel = topk_indices(w_ref, kt)   # the oracle's own set for the reuse layer
        o1_ref, _ = A.sparse_prefill_tile(Q1, K1, V1, sel, 0, h, t, gm, scale)
        check_out(outs[1][0, h, r0:r1], o1_ref, what=("reuse rows", h, t))
