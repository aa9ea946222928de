"""The seeded generator: deterministic bytes, N(0,1)-like moments, planted
keys visible in the exact Top-k, and the cross-layer chain."""
import hashlib

import numpy as np
import torch

from long_context_anchor_gb300 import configs
from long_context_anchor_gb300.workloads import make_layers, layer_rhos
from oracle import attention as A


def _digest(ts):
    h = hashlib.sha256()
    for t in ts:
        h.update(t.contiguous().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()


def test_same_seed_same_bytes():
    w = configs.TINY_DECODE
    a = make_layers(w)
    b = make_layers(w)
    for x, y in zip(a, b):
        assert _digest(x) == _digest(y)
    c = make_layers(w, seed=w.seed + 1)
    assert _digest(a[1]) != _digest(c[1])


def test_moments_and_chain():
    w = configs.TINY_DECODE.with_(n_layers=3, n_plants=0)
    qs, ks, vs = make_layers(w)
    for x in ks + vs:
        assert abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1) < 0.05
    corr = float((ks[0] * ks[1]).mean() / (ks[0].std() * ks[1].std()))
    assert abs(corr - 0.9) < 0.03


def test_planted_keys_surface_in_topk():
    w = configs.TINY_DECODE
    qs, ks, vs = make_layers(w)
    q, k, v = (x.double().numpy() for x in (qs[0], ks[0], vs[0]))
    _, idx, s = A.anchor_decode(q, k, v, w.topk)
    # planted keys score about 3 above the N(0,1) bulk: most of the 16 are selected
    gm = A.default_group_map(w.n_q_heads, w.n_kv_heads)
    for h in range(w.n_q_heads):
        qd = q[0, h] / np.linalg.norm(q[0, h])
        proj = k[0, gm[h]] @ qd
        planted = np.argsort(-proj)[:16]
        assert len(set(planted.tolist()) & set(idx[0, h].tolist())) >= 12


def test_bf16_storage_and_sink():
    w = configs.LLAMA8B_DECODE_32K.with_(n_layers=2, batch=1, kv_len=256, topk=32)
    qs, ks, vs = make_layers(w)
    assert qs[0].dtype == torch.bfloat16 and ks[0].shape == (1, 8, 256, 128)
    # the sink adds exactly 4 * u_g to key 0 (u_g: normalised sum of the group's queries)
    w32 = w.with_(dtype="f32")
    with_sink = make_layers(w32)[1][0]
    without = make_layers(w32.with_(sink=False))[1][0]
    diff = with_sink - without
    q = make_layers(w32)[0][0][0]
    for g in range(8):
        u = q[4 * g:4 * g + 4].sum(0)
        torch.testing.assert_close(diff[0, g, 0], 4 * u / u.norm(), rtol=0, atol=1e-5)
    assert float(diff[0, :, 1:].abs().max()) == 0.0


def test_rho_range():
    r = layer_rhos(configs.SWEEP_CALIBRATION)
    assert len(r) == 32 and all(0.7 <= x <= 0.95 for x in r)
    assert r == layer_rhos(configs.SWEEP_CALIBRATION)


def test_sweep_evaluation_shares_calibration_rhos():
    """The sweep's evaluation sequences are fresh draws (other seeds) on the
    calibration's per-layer chain coefficients."""
    cal = layer_rhos(configs.SWEEP_CALIBRATION)
    assert layer_rhos(configs.SWEEP_DECODE) == cal
    for n in configs.SWEEP_PREFILL_LENGTHS:
        w = configs.sweep_prefill(n)
        assert layer_rhos(w) == cal and w.seed != configs.SWEEP_CALIBRATION.seed
        assert w.topk == n // 8 and w.kv_len == n
    assert configs.SWEEP_DECODE.seed != configs.SWEEP_CALIBRATION.seed
