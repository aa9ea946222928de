"""GPU parity of GQA-pooled index sets (one set per KV head) against the
float64 oracle, through the C ABI: pooled anchor decode (group sums of the
softmax weights, their Top-k), reuse decode over the group sets, pooled
anchor / reuse prefill, the stack driver, and sampled checks at full size.

Pooled weights are probabilities (they sum to the group size), so near-ties
are judged on their logarithm: an index that differs from the oracle's set
must have log w within 1e-3 of the oracle's k-th log-weight (the same
tolerance the per-head sets get on the logit scale)."""
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
                         packed_tile)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None
# relative error of a pooled weight: the fp32 logits differ from the
# oracle's by up to 1e-3 (absolute), which moves exp(s) by up to ~1e-3
W_REL = 2e-3


@pytest.fixture(scope="module")
def K():
    __graft_entry__.build()
    from long_context_anchor_gb300 import kascade
    return kascade


def _rand_layer(B, Hq, Hkv, N, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, d, generator=g)
    k = torch.randn(B, Hkv, N, d, generator=g)
    v = torch.randn(B, Hkv, N, d, generator=g)
    return [x.to(dtype).to(DEV) for x in (q, k, v)]


def _dev_idx(idx):
    """Oracle index sets as the int32 device tensor the library takes."""
    return torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to(DEV)


def _prefill_layer(B, Hq, Hkv, N, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(B, H, N, 128, generator=g).to(torch.bfloat16).to(DEV)
            for H in (Hq, Hkv, Hkv)]


def _log(w):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(w, dtype=np.float64))


def _check_weights(got, ref, what="pooled weights"):
    g = f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    assert g.shape == ref.shape and np.isfinite(g).all(), what
    err = np.abs(g - ref)
    assert (err <= W_REL * ref + 1e-9).all(), (what, float((err / (ref + 1e-30)).max()))


SHAPES = [  # B, Hq, Hkv, N, d, dtype
    (1, 4, 2, 512, 64, torch.float32),
    (1, 4, 2, 512, 64, torch.bfloat16),
    (2, 8, 8, 1000, 128, torch.bfloat16),     # G = 1: pooled = per head
    (2, 16, 2, 4097, 64, torch.bfloat16),     # G = 8, ragged
    (3, 8, 2, 3000, 128, torch.bfloat16),     # G = 4
    (1, 4, 2, 70, 128, torch.bfloat16),       # shorter than one split
]


@pytest.mark.parametrize("shape", SHAPES)
def test_pooled_anchor_decode_matches_oracle(K, shape):
    B, Hq, Hkv, N, d, dt = shape
    q, k, v = _rand_layer(B, Hq, Hkv, N, d, dt, seed=N + 3 * Hq)
    topk = max(1, N // 8)
    out, idx, w = K.anchor_decode(q, k, v, topk, return_scores=True, pooled=True)
    assert idx.shape == (B, Hkv, topk) and w.shape == (B, Hkv, N)
    o_ref, _, w_ref = A.anchor_decode_pooled(f64(q), f64(k), f64(v), topk)
    tight = dt == torch.float32
    check_out(out, o_ref, *((1e-4, 1e-5) if tight else (2e-2, 2e-3)))
    _check_weights(w, w_ref)
    got, wg = idx.cpu().numpy(), w.cpu().numpy()
    for b in range(B):
        for g in range(Hkv):
            check_index_set(got[b, g], _log(w_ref[b, g]), topk)
            # bit-exact against the oracle rule on the kernel's own fp32 weights
            assert got[b, g].tolist() == topk_indices(wg[b, g], topk).tolist()
    if Hq == Hkv:   # one head per group: the per-head sets, up to fp32 ties of exp
        _, idx_h = K.anchor_decode(q, k, v, topk)
        ih = idx_h.cpu().numpy()
        for b in range(B):
            for g in range(Hkv):
                assert len(set(ih[b, g].tolist()) ^ set(got[b, g].tolist())) <= 2


@pytest.mark.parametrize("shape", SHAPES)
def test_pooled_reuse_decode_matches_oracle(K, shape):
    B, Hq, Hkv, N, d, dt = shape
    q, k, v = _rand_layer(B, Hq, Hkv, N, d, dt, seed=5 * N + Hq)
    topk = max(1, N // 8)
    _, idx_ref, _ = A.anchor_decode_pooled(f64(q), f64(k), f64(v), topk)   # the oracle's sets
    q2, k2, v2 = _rand_layer(B, Hq, Hkv, N, d, dt, seed=13 * N + Hq)
    out = K.reuse_decode(q2, k2, v2, _dev_idx(idx_ref), pooled=True)
    o_ref = A.sparse_decode_pooled(f64(q2), f64(k2), f64(v2), idx_ref)
    check_out(out, o_ref, *((1e-4, 1e-5) if dt == torch.float32 else (2e-2, 2e-3)))


def test_pooled_permuted_group_map(K):
    gm = [1, 0, 3, 2, 0, 1, 2, 3]
    q, k, v = _rand_layer(2, 8, 4, 777, 128, torch.bfloat16, seed=15)
    out, idx, w = K.anchor_decode(q, k, v, 50, group_map=gm, return_scores=True, pooled=True)
    o_ref, _, w_ref = A.anchor_decode_pooled(f64(q), f64(k), f64(v), 50, gm)
    check_out(out, o_ref)
    _check_weights(w, w_ref)
    got = idx.cpu().numpy()
    for b in range(2):
        for g in range(4):
            check_index_set(got[b, g], _log(w_ref[b, g]), 50)
    _, idx_ref, _ = A.anchor_decode_pooled(f64(q), f64(k), f64(v), 50, gm)
    out_r = K.reuse_decode(q, k, v, _dev_idx(idx_ref), group_map=gm, pooled=True)
    check_out(out_r, A.sparse_decode_pooled(f64(q), f64(k), f64(v), idx_ref, gm))


def test_pooled_reuse_poison_outside_group_sets(K):
    B, Hq, Hkv, N, d = 2, 8, 2, 2048, 128
    q, k, v = _rand_layer(B, Hq, Hkv, N, d, torch.bfloat16, seed=17)
    _, idx = K.anchor_decode(q, k, v, 200, pooled=True)
    out = K.reuse_decode(q, k, v, idx, pooled=True)
    used = torch.zeros(B, Hkv, N, dtype=torch.bool, device=DEV)
    used.scatter_(2, idx.long(), True)
    kp, vp = k.clone(), v.clone()
    kp[~used] = float("nan")
    vp[~used] = float("nan")
    assert torch.equal(K.reuse_decode(q, kp, vp, idx, pooled=True), out)


def test_pooled_nan_logit_reported(K):
    ws = K.Workspace(DEV)
    q, k, v = _rand_layer(1, 4, 2, 512, 64, torch.float32, seed=19)
    k[0, 1, 33, 5] = float("nan")
    K.anchor_decode(q, k, v, 16, ws=ws, pooled=True)
    assert ws.device_error() == K.BAD_INPUT
    K.anchor_decode(q, k.nan_to_num(0.0), v, 16, ws=ws, pooled=True)
    assert ws.device_error() == K.OK


@pytest.mark.parametrize("bad", ["out_of_range", "negative", "not_ascending", "repeated"])
def test_pooled_reuse_decode_bad_set_reported(K, bad):
    """Pooled sets are gathered as they are (no plan); an entry outside
    [0, N), or a set that does not strictly ascend, is reported as bad input
    and the entry is not read; a valid set afterwards reports nothing."""
    ws = K.Workspace(DEV)
    B, Hq, Hkv, N, topk = 2, 8, 2, 3000, 100
    q, k, v = _rand_layer(B, Hq, Hkv, N, 128, torch.bfloat16, seed=23)
    rng = np.random.default_rng(3)
    idx = np.stack([np.stack([np.sort(rng.choice(N, topk, replace=False)) for _ in range(Hkv)])
                    for _ in range(B)]).astype(np.int32)
    good = _dev_idx(idx)
    if bad == "out_of_range":
        idx[1, 0, -1] = N
    elif bad == "negative":
        idx[0, 1, 0] = -5
    elif bad == "not_ascending":
        idx[0, 0, 10], idx[0, 0, 11] = idx[0, 0, 11], idx[0, 0, 10]
    else:
        idx[1, 1, 40] = idx[1, 1, 39]
    K.reuse_decode(q, k, v, _dev_idx(idx), ws=ws, pooled=True)
    assert ws.device_error() == K.BAD_INPUT
    out = K.reuse_decode(q, k, v, good, ws=ws, pooled=True)
    assert ws.device_error() == K.OK
    check_out(out, A.sparse_decode_pooled(f64(q), f64(k), f64(v), good.cpu().numpy()))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pooled_decode_stack_matches_layer_calls(K, dtype):
    w = configs.TINY_DECODE.with_(dtype=dtype, n_layers=4, anchors=(0, 2))
    qs, ks, vs = make_layers(w)
    dq, dk, dv = ([x.to(DEV) for x in xs] for xs in (qs, ks, vs))
    outs, idx_buf = K.run_stack(K.DECODE, dq, dk, dv, w.topk, list(w.anchors), pooled=True)
    o0, i0 = K.anchor_decode(dq[0], dk[0], dv[0], w.topk, pooled=True)
    o1 = K.reuse_decode(dq[1], dk[1], dv[1], i0, pooled=True)
    o2, i2 = K.anchor_decode(dq[2], dk[2], dv[2], w.topk, pooled=True)
    o3 = K.reuse_decode(dq[3], dk[3], dv[3], i2, pooled=True)
    for a_, b_ in zip(outs, [o0, o1, o2, o3]):
        assert torch.equal(a_, b_)
    assert idx_buf.shape == (w.batch, w.n_kv_heads, w.topk) and torch.equal(idx_buf, i2)
    # against the oracle stack, which selects its own float64 pooled sets
    ref_outs, _, _ = run_oracle_stack("decode", [(f64(a_), f64(b_), f64(c_))
                                                 for a_, b_, c_ in zip(qs, ks, vs)],
                                      w.topk, list(w.anchors), pooled=True)
    for o, r in zip(outs, ref_outs):
        check_out(o, r)


# ----------------------------------------------------------------- prefill --

@pytest.mark.parametrize("shape,topk", [((1, 4, 2, 300), 64), ((2, 8, 2, 520), 130),
                                        ((1, 8, 1, 1024), 128), ((1, 2, 2, 384), 100)])
def test_pooled_anchor_prefill_matches_oracle(K, shape, topk):
    B, Hq, Hkv, N = shape
    q, k, v = _prefill_layer(B, Hq, Hkv, N, seed=3 * N + topk)
    out, idx, wts = K.anchor_prefill(q, k, v, topk, pooled=True, return_weights=True)
    nT = A.n_tiles(N)
    assert idx.shape == (B, Hkv, nT, topk)
    assert wts.shape == (B, Hkv, K.packed_tile_len(N))
    Q, Kh, V = f64(q), f64(k), f64(v)
    gm = A.default_group_map(Hq, Hkv)
    check_out(out, A.dense_prefill(Q, Kh, V))
    got = idx.cpu().numpy()
    w_gpu = wts.cpu().numpy()
    scale = 1.0 / np.sqrt(128)
    for b in range(B):
        for g in range(Hkv):
            for t in range(nT):
                w = A.tile_weights_pooled(Q, Kh, b, g, t, gm, scale)
                w_row = packed_tile(w_gpu[b, g], t, N)
                check_weights(w_row, w, what=("pooled tile weights", b, g, t))
                kt = min(topk, w.shape[0])
                row = got[b, g, t]
                check_topk_exact(row, w_row, kt, what=("pooled tile top-k", b, g, t))
                check_index_set(row[:kt], _log(w), kt, what=("pooled tile set", b, g, t))


@pytest.mark.parametrize("shape,topk", [((1, 4, 2, 300), 64), ((2, 8, 2, 520), 130)])
def test_pooled_reuse_prefill_matches_oracle(K, shape, topk):
    B, Hq, Hkv, N = shape
    q, k, v = _prefill_layer(B, Hq, Hkv, N, seed=7 * N + 1)
    _, idx_ref = A.anchor_prefill_pooled(f64(q), f64(k), f64(v), topk)   # the oracle's sets
    q2, k2, v2 = _prefill_layer(B, Hq, Hkv, N, seed=9 * N + 1)
    out = K.reuse_prefill(q2, k2, v2, _dev_idx(idx_ref), pooled=True)
    check_out(out, A.sparse_prefill_pooled(f64(q2), f64(k2), f64(v2), idx_ref))


@pytest.mark.parametrize("shape,topk", [((1, 4, 2, 640), 200), ((1, 16, 2, 384), 96),
                                        ((2, 4, 1, 300), 64)])
def test_pooled_reuse_prefill_equals_per_head_kernel(K, shape, topk):
    # the paired-head kernel (two heads of a KV head per CTA, one gather)
    # against the per-head kernel given each head its group's set
    B, Hq, Hkv, N = shape
    q, k, v = _prefill_layer(B, Hq, Hkv, N, seed=11 * N + Hq)
    _, idx_ref = A.anchor_prefill_pooled(f64(q), f64(k), f64(v), topk)   # the oracle's sets
    idx = _dev_idx(idx_ref)
    out_p = K.reuse_prefill(q, k, v, idx, pooled=True)
    gm = default_gmap(Hq, Hkv)
    idx_h = idx[:, gm].contiguous()
    out_h = K.reuse_prefill(q, k, v, idx_h)
    assert (out_p.float() - out_h.float()).abs().max().item() <= 1.6e-2
    check_out(out_p, A.sparse_prefill_pooled(f64(q), f64(k), f64(v), idx_ref))


def test_pooled_reuse_prefill_poison_and_empty_rows(K):
    B, Hq, Hkv, N, topk = 1, 8, 2, 512, 64
    q, k, v = _prefill_layer(B, Hq, Hkv, N, seed=23)
    nT = A.n_tiles(N)
    rng = np.random.default_rng(5)
    idx = np.full((B, Hkv, nT, topk), -1, dtype=np.int32)
    for g in range(Hkv):
        for t in range(nT):
            L = min(N, 128 * (t + 1))
            # no saved key below position 30: rows 0..29 see an empty set
            sel = np.sort(rng.choice(np.arange(30, L), min(topk, L - 30), replace=False))
            idx[0, g, t, :sel.size] = sel
    idx_t = torch.from_numpy(idx).to(DEV)
    out = K.reuse_prefill(q, k, v, idx_t, pooled=True)
    check_out(out, A.sparse_prefill_pooled(f64(q), f64(k), f64(v), idx))
    assert float(out[0, :, :30].float().abs().max()) == 0.0
    used = torch.zeros(B, Hkv, N, dtype=torch.bool, device=DEV)
    for g in range(Hkv):
        sel = idx_t[0, g].reshape(-1)
        used[0, g, sel[sel >= 0].long()] = True
    kp, vp = k.clone(), v.clone()
    kp[~used] = float("nan")
    vp[~used] = float("nan")
    assert torch.equal(K.reuse_prefill(q, kp, vp, idx_t, pooled=True), out)


def test_pooled_reuse_prefill_bad_index_reported(K):
    ws = K.Workspace(DEV)
    q, k, v = _prefill_layer(1, 4, 2, 256, seed=29)
    idx = torch.arange(32, dtype=torch.int32, device=DEV).expand(1, 2, 2, 32).contiguous()
    idx[0, 1, 1, 7] = 4096
    K.reuse_prefill(q, k, v, idx, ws=ws, pooled=True)
    assert ws.device_error() == K.BAD_INPUT


def test_pooled_prefill_stack_matches_layer_calls(K):
    w = configs.LLAMA8B_PREFILL_16K.with_(n_layers=3, kv_len=640, topk=80, anchors=(0,))
    qs, ks, vs = make_layers(w, device=DEV)
    outs, idx_buf = K.run_stack(K.PREFILL, qs, ks, vs, w.topk, [0], pooled=True)
    o0, i0 = K.anchor_prefill(qs[0], ks[0], vs[0], w.topk, pooled=True)
    o1 = K.reuse_prefill(qs[1], ks[1], vs[1], i0, pooled=True)
    o2 = K.reuse_prefill(qs[2], ks[2], vs[2], i0, pooled=True)
    for a_, b_ in zip(outs, [o0, o1, o2]):
        assert torch.equal(a_, b_)
    assert torch.equal(idx_buf, i0)
    # against the oracle stack, which selects its own float64 pooled tile sets
    ref_outs, _, _ = run_oracle_stack("prefill", [(f64(a_), f64(b_), f64(c_))
                                                  for a_, b_, c_ in zip(qs, ks, vs)],
                                      w.topk, [0], pooled=True)
    for o, r in zip(outs, ref_outs):
        check_out(o, r)


# -------------------------------------------------------- full-size samples --

def test_full_size_pooled_decode_sampled(K):
    w = configs.LLAMA8B_DECODE_32K.with_(n_layers=2)
    qs, ks, vs = make_layers(w, device=DEV)
    outs, idx = K.run_stack(K.DECODE, qs, ks, vs, w.topk, [0], pooled=True)
    torch.cuda.synchronize()
    gm = default_gmap(w.n_q_heads, w.n_kv_heads)
    scale = 1.0 / np.sqrt(w.head_dim)
    idx_np = idx.cpu().numpy()
    for b in (0, w.batch - 1):
        q0 = f64(qs[0][b:b + 1])
        K0, V0 = f64(ks[0][b:b + 1]), f64(vs[0][b:b + 1])
        s = A.decode_logits(q0, K0, gm, scale)
        wp = A.pooled_decode_weights(s, gm, w.n_kv_heads)[0]
        for g in (0, 3, w.n_kv_heads - 1):
            check_index_set(idx_np[b, g], _log(wp[g]), w.topk, what="pooled set")
        for h in (0, 13, w.n_q_heads - 1):
            sel = topk_indices(wp[gm[h]], w.topk)   # the oracle's own set for the reuse layer
            o_ref = A.sparse_decode_pooled(f64(qs[1][b:b + 1, h:h + 1]),
                                           f64(ks[1][b:b + 1, gm[h]:gm[h] + 1]),
                                           f64(vs[1][b:b + 1, gm[h]:gm[h] + 1]),
                                           sel[None, None, :], [0])[0, 0]
            check_out(outs[1][b, h], o_ref, what="pooled reuse row")


def test_full_size_pooled_prefill_sampled(K):
    w = configs.LLAMA8B_PREFILL_16K.with_(n_layers=2)
    qs, ks, vs = make_layers(w, device=DEV)
    outs, idx = K.run_stack(K.PREFILL, qs, ks, vs, w.topk, [0], pooled=True)
    _, idx_a, wts = K.anchor_prefill(qs[0], ks[0], vs[0], w.topk, pooled=True,
                                     return_weights=True)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_a)
    gm = default_gmap(w.n_q_heads, w.n_kv_heads)
    scale = 1.0 / np.sqrt(w.head_dim)
    nT = A.n_tiles(w.kv_len)
    idx_np = idx.cpu().numpy()
    for g, t in [(0, 0), (w.n_kv_heads - 1, nT - 1), (3, 40)]:
        heads = [h for h in range(w.n_q_heads) if gm[h] == g]
        L = A.prefix_len(t, w.kv_len)
        Qg = qs[0][:, heads, :L].float().cpu().numpy()
        Kg = ks[0][:, g:g + 1, :L].float().cpu().numpy()
        wt = A.tile_weights_pooled(Qg, Kg, 0, 0, t, [0] * len(heads), scale)
        w_row = packed_tile(wts[0, g].cpu().numpy(), t, w.kv_len)
        check_weights(w_row, wt, what=("pooled tile weights", g, t))
        kt = min(w.topk, L)
        check_topk_exact(idx_np[0, g, t], w_row, kt, what=("pooled tile top-k", g, t))
        check_index_set(idx_np[0, g, t, :kt], _log(wt), kt, what="pooled tile set")
        # reuse rows of one head of the group over the group's set
        h = heads[1]
        r0, r1 = A.tile_rows(t, w.kv_len)
        sel = topk_indices(wt, kt)   # the oracle's own set for the reuse layer
        Q1 = qs[1][:, h:h + 1, :L].float().cpu().numpy()
        K1 = ks[1][:, g:g + 1, :L].float().cpu().numpy()
        V1 = vs[1][:, g:g + 1, :L].float().cpu().numpy()
        o_ref, _ = A.sparse_prefill_tile(Q1, K1, V1, sel, 0, 0, t, [0], scale)
        check_out(outs[1][0, h, r0:r1], o_ref, what="pooled reuse rows")
