"""GPU edge cases of the path against the float64 oracle, through the C ABI:
an empty Top-k, k = 1 and k = N, a single cached key, a sequence shorter than
one prefill tile (down to a single row), and a single-key reuse set (whose
output is that key's value row)."""
import numpy as np
import pytest
import torch

import __graft_entry__
from oracle import attention as A
from oracle.topk import topk_indices
from gpu_helpers import check_topk_exact, check_weights, log_w, packed_tile, check_index_set, check_out, f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def K():
    __graft_entry__.build()
    from long_context_anchor_gb300 import kascade
    return kascade


def _dev_idx(idx):
    return torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to(DEV)


def _decode_layer(B, Hq, Hkv, N, d, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(*shape, generator=g).to(dtype).to(DEV)
            for shape in ((B, Hq, d), (B, Hkv, N, d), (B, Hkv, N, d))]


def _prefill_layer(B, Hq, Hkv, N, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(B, H, N, 128, generator=g).to(torch.bfloat16).to(DEV)
            for H in (Hq, Hkv, Hkv)]


def test_topk_empty_and_extreme_k(K):
    ws = K.Workspace(DEV)
    empty = torch.empty(0, 100, device=DEV)
    assert K.topk(empty, 5, ws=ws).shape == (0, 5)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 777)).astype(np.float32)
    x[2, 100:200] = 0.5                      # ties
    xt = torch.from_numpy(x).to(DEV)
    for k in (1, 2, 776, 777):
        got = K.topk(xt, k, ws=ws).cpu().numpy()
        for r in range(5):
            assert got[r].tolist() == topk_indices(x[r], k).tolist(), (k, r)
    assert ws.device_error() == K.OK


@pytest.mark.parametrize("N", [1, 70, 1000])
def test_decode_k_one_and_k_n(K, N):
    B, Hq, Hkv, d = 2, 8, 2, 128
    q, k, v = _decode_layer(B, Hq, Hkv, N, d, seed=N)
    Q, Kh, V = f64(q), f64(k), f64(v)
    for topk in sorted({1, N}):
        out, idx, s = K.anchor_decode(q, k, v, topk, return_scores=True)
        o_ref, _, s_ref = A.anchor_decode(Q, Kh, V, topk)
        check_out(out, o_ref)
        got, sc = idx.cpu().numpy(), s.cpu().numpy()
        for b in range(B):
            for h in range(Hq):
                check_index_set(got[b, h], s_ref[b, h], topk)
                assert got[b, h].tolist() == topk_indices(sc[b, h], topk).tolist()
        if topk == N:
            assert (got == np.arange(N)).all()
    # a single-key set: the output is that key's value row
    _, idx1, _ = A.anchor_decode(Q, Kh, V, 1)
    out1 = K.reuse_decode(q, k, v, _dev_idx(idx1))
    gm = A.default_group_map(Hq, Hkv)
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_allclose(f64(out1[b, h]), V[b, gm[h], idx1[b, h, 0]], atol=1e-2)
    check_out(out1, A.sparse_decode(Q, Kh, V, idx1))


@pytest.mark.parametrize("N", [1, 70, 129, 333])
def test_prefill_shorter_than_a_tile_and_ragged(K, N):
    """Rows shorter than a tile and ragged last tiles; the packed tile weights
    then start off 16-byte boundaries for every (sequence, head) after the
    first (their row length is not a multiple of 4)."""
    B, Hq, Hkv = 1, 4, 2
    q, k, v = _prefill_layer(B, Hq, Hkv, N, seed=7 + N)
    Q, Kh, V = f64(q), f64(k), f64(v)
    check_out(K.dense_prefill(q, k, v), A.dense_prefill(Q, Kh, V))
    gm = A.default_group_map(Hq, Hkv)
    scale = 1.0 / np.sqrt(128)
    for topk in sorted({1, min(N, 40), N}):
        out, idx, wts = K.anchor_prefill(q, k, v, topk, return_weights=True)
        o_ref, idx_ref = A.anchor_prefill(Q, Kh, V, topk)
        check_out(out, o_ref)
        got, w_gpu = idx.cpu().numpy(), wts.cpu().numpy()
        for h in range(Hq):
            for t in range(A.n_tiles(N)):
                w = A.tile_weights(Q, Kh, 0, h, t, gm, scale)
                w_row = packed_tile(w_gpu[0, h], t, N)
                check_weights(w_row, w, what=("tile weights", h, t))
                kt = min(topk, w.shape[0])
                check_topk_exact(got[0, h, t], w_row, kt, what=("tile top-k", h, t))
                check_index_set(got[0, h, t, :kt], log_w(w), kt)
        out_r = K.reuse_prefill(q, k, v, _dev_idx(idx_ref))
        check_out(out_r, A.sparse_prefill(Q, Kh, V, idx_ref))
        # pooled sets: the group sums of the same weights
        _, idx_p, wts_p = K.anchor_prefill(q, k, v, topk, return_weights=True, pooled=True)
        gp, wp = idx_p.cpu().numpy(), wts_p.cpu().numpy()
        for g in range(Hkv):
            for t in range(A.n_tiles(N)):
                w = A.tile_weights_pooled(Q, Kh, 0, g, t, gm, scale)
                w_row = packed_tile(wp[0, g], t, N)
                check_weights(w_row, w, what=("pooled tile weights", g, t))
                check_topk_exact(gp[0, g, t], w_row, min(topk, w.shape[0]), what=("pooled", g, t))
