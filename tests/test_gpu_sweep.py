"""GPU parity at the schedule-sweep sizes (the 32-layer Llama-3.1-8B attention
shape): calibration on 4 sequences of 32768 keys with every layer run as an
anchor, the anchor DP's six anchors, then the decode stack at batch 16
(N = 32768, k = 4096) and the prefill stack at N = 65536 (k = 8192, 512
tiles) run with those anchors, checked on sampled units against the oracle.
The anchor DP and the cross-layer overlap follow the euno.news summary,
Methodology 4, and the opentrain.ai Abstract (anchors chosen by a dynamic
programme over cross-layer similarity)."""
import numpy as np
import pytest
import torch

import __graft_entry__
from long_context_anchor_gb300 import configs
from long_context_anchor_gb300.workloads import make_layers, group_map as default_gmap
from oracle import attention as A
from oracle.schedule import objective, overlap_similarity, schedule_anchors as oracle_dp
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


@pytest.fixture(scope="module")
def calibration(K):
    """Calibration at full size: the kernel's similarity and sets, the oracle's
    own float64 sets, their similarity, and per layer the number of set
    positions where the kernel's sets and the oracle's differ (near-ties)."""
    w = configs.SWEEP_CALIBRATION
    L, B, Hq, N, k = w.n_layers, w.batch, w.n_q_heads, w.kv_len, w.topk
    qs, ks, vs = make_layers(w, device=DEV)
    sim, sets = K.calibrate(qs, ks, vs, k)
    sets_np = sets.cpu().numpy().reshape(L, B * Hq, k)
    gm = default_gmap(Hq, w.n_kv_heads)
    scale = 1.0 / np.sqrt(w.head_dim)
    own, swaps = [], []
    for layer in range(L):
        rows = A.decode_logits(f64(qs[layer]), f64(ks[layer]), gm, scale).reshape(B * Hq, N)
        own.append(np.stack([topk_indices(rows[u], k) for u in range(B * Hq)]))
        swaps.append(sum(check_index_set(sets_np[layer, u], rows[u], k,
                                         what=("calibration set", layer, u)) // 2
                         for u in range(B * Hq)))
    del qs, ks, vs
    torch.cuda.empty_cache()
    return np.array(sim), sets_np, overlap_similarity(own, k), swaps


@pytest.fixture(scope="module")
def anchors(K, calibration):
    sim = calibration[0]
    a, _ = K.schedule_anchors(sim.tolist(), configs.SWEEP_N_ANCHORS)
    return a


def test_sweep_calibration_and_dp(K, calibration, anchors):
    sim, sets_np, ref, swaps = calibration
    w = configs.SWEEP_CALIBRATION
    L, U, k = w.n_layers, w.batch * w.n_q_heads, w.topk
    # the similarity is the exact overlap arithmetic on the kernel's own sets
    np.testing.assert_allclose(sim, overlap_similarity(list(sets_np), k), rtol=0, atol=1e-12)
    # against the oracle's sets: each swapped position moves |S_i ∩ S_l| by one
    bound = (np.add.outer(swaps, swaps)) / (U * k) + 1e-12
    assert (np.abs(sim - ref) <= bound).all(), float(np.abs(sim - ref).max())
    # the C DP is the oracle DP on the same matrix
    m = configs.SWEEP_N_ANCHORS
    ao, fo = oracle_dp(sim, m)
    assert anchors == ao
    assert len(anchors) == m and anchors[0] == 0
    # and near-optimal under the oracle's own similarity
    _, f_ref = oracle_dp(ref, m)
    assert objective(ref, anchors) >= f_ref - 2 * L * float(bound.max())


def _decode_unit_host(qs, ks, vs, layer, b, h, g):
    """One (sequence, query head) of one layer on the host, mapped to index 0."""
    return (f64(qs[layer][b:b + 1, h:h + 1]), f64(ks[layer][b:b + 1, g:g + 1]),
            f64(vs[layer][b:b + 1, g:g + 1]))


def _owner(anchors, layer):
    return max(a for a in anchors if a <= layer)


def test_sweep_decode_b16_through_dp_anchors(K, anchors):
    w = configs.SWEEP_DECODE
    L = w.n_layers
    qs, ks, vs = make_layers(w, device=DEV)
    outs, idx = K.run_stack(K.DECODE, qs, ks, vs, w.topk, anchors)
    torch.cuda.synchronize()
    # the last anchor's sets, bit-exact on its own fp32 logits
    last = anchors[-1]
    _, idx_a, s_gpu = K.anchor_decode(qs[last], ks[last], vs[last], w.topk, return_scores=True)
    assert torch.equal(idx, idx_a)
    gm = default_gmap(w.n_q_heads, w.n_kv_heads)
    scale = 1.0 / np.sqrt(w.head_dim)
    rng = np.random.default_rng(16)
    layers = sorted({anchors[0], anchors[1], anchors[1] + 1, last, L - 1})
    for layer in layers:
        owner = _owner(anchors, layer)
        units = [(0, 0), (w.batch - 1, w.n_q_heads - 1),
                 (int(rng.integers(w.batch)), int(rng.integers(w.n_q_heads)))]
        for b, h in units:
            g = gm[h]
            o_a, sel, s_ref = A.decode_unit(*_decode_unit_host(qs, ks, vs, owner, b, h, g),
                                            0, 0, w.topk, [0], scale)
            if layer == owner:
                check_out(outs[layer][b, h], o_a, what=("anchor out", layer, b, h))
            else:
                o_r = A.decode_unit(*_decode_unit_host(qs, ks, vs, layer, b, h, g),
                                    0, 0, w.topk, [0], scale, idx=sel)
                check_out(outs[layer][b, h], o_r, what=("reuse out", layer, b, h))
            if owner == last:
                got = idx[b, h].cpu().numpy()
                check_topk_exact(got, s_gpu[b, h].cpu().numpy(), w.topk, what=("top-k", b, h))
                check_index_set(got, s_ref, w.topk, what=("set", b, h))


def test_sweep_prefill_n65536_through_dp_anchors(K, anchors):
    w = configs.sweep_prefill(65536)
    L, N = w.n_layers, w.kv_len
    qs, ks, vs = make_layers(w, device=DEV)
    outs, idx = K.run_stack(K.PREFILL, qs, ks, vs, w.topk, anchors)
    last = anchors[-1]
    _, idx_a, wts = K.anchor_prefill(qs[last], ks[last], vs[last], w.topk, return_weights=True)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_a)
    gm = default_gmap(w.n_q_heads, w.n_kv_heads)
    scale = 1.0 / np.sqrt(w.head_dim)
    nT = A.n_tiles(N)
    rng = np.random.default_rng(65)
    idx_np = idx.cpu().numpy()
    for layer in sorted({anchors[0], last, last + 1, L - 1}):
        owner = _owner(anchors, layer)
        for h, t in [(0, 0), (w.n_q_heads - 1, nT - 1),
                     (int(rng.integers(w.n_q_heads)), int(rng.integers(nT)))]:
            g = gm[h]
            Lt = A.prefix_len(t, N)
            r0, r1 = A.tile_rows(t, N)
            host = lambda lay: (f64(qs[lay][:, h:h + 1, :Lt]), f64(ks[lay][:, g:g + 1, :Lt]),
                                f64(vs[lay][:, g:g + 1, :Lt]))
            Qo, Ko, Vo = host(owner)
            w_ref = A.tile_weights(Qo, Ko, 0, 0, t, [0], scale)
            kt = min(w.topk, Lt)
            if layer == owner:
                o_ref, _ = A.dense_prefill_tile(Qo, Ko, Vo, 0, 0, t, [0], scale)
                check_out(outs[layer][0, h, r0:r1], o_ref, what=("anchor rows", layer, h, t))
            else:
                sel = topk_indices(w_ref, kt)   # the oracle's own set for the reuse layer
                Q1, K1, V1 = host(layer)
                o_ref, _ = A.sparse_prefill_tile(Q1, K1, V1, sel, 0, 0, t, [0], scale)
                check_out(outs[layer][0, h, r0:r1], o_ref, what=("reuse rows", layer, h, t))
            if owner == last:
                w_row = packed_tile(wts[0, h].cpu().numpy(), t, N)
                check_weights(w_row, w_ref, what=("tile weights", h, t))
                check_topk_exact(idx_np[0, h, t], w_row, kt, what=("tile top-k", h, t))
                check_index_set(idx_np[0, h, t, :kt], log_w(w_ref), kt, what=("tile set", h, t))
