"""GPU checks of the anchor-selection path: the cross-layer overlap kernel
against exact set arithmetic, calibration (every layer as an anchor) against
the oracle's overlap similarity, and the C DP against the oracle DP."""
import numpy as np
import pytest
import torch

import __graft_entry__
from long_context_anchor_gb300 import configs
from long_context_anchor_gb300.workloads import make_layers
from oracle import attention as A
from oracle.schedule import overlap_similarity, schedule_anchors as oracle_dp
from gpu_helpers import check_index_set

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def K():
    __graft_entry__.build()
    from long_context_anchor_gb300 import kascade
    return kascade


def test_layer_overlap_exact(K):
    rng = np.random.default_rng(0)
    L, U, k, nb = 5, 7, 50, 1000
    sets = np.stack([np.stack([np.sort(rng.choice(nb, k, replace=False)) for _ in range(U)])
                     for _ in range(L)]).astype(np.int32)
    counts = K.layer_overlap(torch.from_numpy(sets).to(DEV), nb).cpu().numpy()
    for i in range(L):
        for l in range(L):
            exp = sum(len(set(sets[i, u]) & set(sets[l, u])) for u in range(U))
            assert counts[i, l] == exp


def test_calibration_and_dp(K):
    w = configs.SWEEP_CALIBRATION.with_(n_layers=6, batch=2, kv_len=2048, topk=256)
    qs, ks, vs = make_layers(w, device=DEV)
    sim, sets = K.calibrate(qs, ks, vs, w.topk)
    sim = np.array(sim)
    sets_np = sets.cpu().numpy()
    # each layer's sets are exactly what the anchor entry point returns
    for layer in range(w.n_layers):
        _, idx = K.anchor_decode(qs[layer], ks[layer], vs[layer], w.topk)
        assert np.array_equal(idx.reshape(-1, w.topk).cpu().numpy(), sets_np[layer])
    # the similarity is the exact overlap arithmetic on the kernel's own sets
    U = w.batch * w.n_q_heads
    np.testing.assert_allclose(sim, overlap_similarity(list(sets_np.reshape(w.n_layers, U, -1)),
                                                       w.topk), rtol=0, atol=1e-12)
    # against the overlap of the oracle's own float64 Top-k sets: the sets may
    # differ only on near-tie keys, and each swapped position moves one
    # intersection count by one
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    own, swaps = [], []
    for layer in range(w.n_layers):
        _, idx, s = A.anchor_decode(f64(qs[layer]), f64(ks[layer]), f64(vs[layer]), w.topk)
        own.append(idx.reshape(-1, w.topk))
        rows = s.reshape(U, -1)
        swaps.append(sum(check_index_set(sets_np[layer].reshape(U, -1)[u], rows[u], w.topk) // 2
                         for u in range(U)))
    ref = overlap_similarity(own, w.topk)
    bound = np.add.outer(swaps, swaps) / (U * w.topk) + 1e-12
    assert (np.abs(sim - ref) <= bound).all()
    from oracle.schedule import objective
    for m in (1, 2, 3, 6):
        # the C DP picks the oracle DP's anchors on the oracle's similarity
        a, f = K.schedule_anchors(ref.tolist(), m)
        ao, fo = oracle_dp(ref, m)
        assert a == ao and abs(f - fo) < 1e-9
        # and, run on the calibrated similarity, a near-optimal schedule under it
        a2, _ = K.schedule_anchors(sim.tolist(), m)
        assert objective(ref, a2) >= fo - 0.05
    # cross-layer correlation makes neighbours overlap more than distant layers
    assert sim[0, 1] > sim[0, 5]


@pytest.mark.parametrize("pooled", [False, True])
def test_recall_calibration_matches_oracle(K, pooled):
    from oracle.schedule import mass_recall_similarity, objective
    w = configs.SWEEP_CALIBRATION.with_(n_layers=6, batch=2, kv_len=2048, topk=256)
    qs, ks, vs = make_layers(w, device=DEV)
    sim, sets = K.calibrate(qs, ks, vs, w.topk, pooled=pooled, similarity="recall")
    sim = np.array(sim)
    L, B, Hq, Hkv = w.n_layers, w.batch, w.n_q_heads, w.n_kv_heads
    gm = A.default_group_map(Hq, Hkv)
    # the sets are the anchor entry point's
    for layer in (0, L - 1):
        _, idx = K.anchor_decode(qs[layer], ks[layer], vs[layer], w.topk, pooled=pooled)
        assert np.array_equal(idx.reshape(-1, w.topk).cpu().numpy(), sets[layer].cpu().numpy())
    # the oracle, on its own float64 softmax and its own Top-k sets
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    probs, own = [], []
    for layer in range(L):
        q, k, v = f64(qs[layer]), f64(ks[layer]), f64(vs[layer])
        if pooled:
            _, idx, _ = A.anchor_decode_pooled(q, k, v, w.topk)
            idx = A.expand_pooled_sets(idx, gm)          # per query head
        else:
            _, idx, _ = A.anchor_decode(q, k, v, w.topk)
        _, s = A.dense_decode(q, k, v)
        probs.append(A.softmax(s).reshape(B * Hq, -1))
        own.append(idx.reshape(B * Hq, w.topk))
    ref = mass_recall_similarity(probs, own)
    for i in range(L):
        for layer in range(L):
            if i <= layer:
                # near-tie set differences move the mass by the tiny gap
                assert abs(sim[i, layer] - ref[i, layer]) < 2e-3, (i, layer)
            else:
                assert sim[i, layer] == 0.0
    # the recall falls with layer distance; the C DP is near-optimal under
    # the oracle's matrix
    assert sim[0, 1] > sim[0, 5]
    for m in (2, 3):
        a, _ = K.schedule_anchors(sim.tolist(), m)
        ao, fo = oracle_dp(ref, m)
        assert objective(ref, a) >= fo - 1e-2
