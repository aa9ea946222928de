"""GPU parity of the decode path (anchor decode + Top-k, reuse decode, dense
decode, the stack driver) against the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import __graft_entry__
from long_context_anchor_gb300 import configs
from long_context_anchor_gb300.workloads import make_layers, group_map as default_gmap
from oracle import attention as A
from oracle.stack import run_stack as run_oracle_stack
from oracle.topk import topk_indices
from gpu_helpers import check_index_set, check_out, check_topk_exact, f64

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


def _rand_layer(B, Hq, Hkv, N, d, dtype, seed, scale_k=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, d, generator=g)
    k = torch.randn(B, Hkv, N, d, generator=g) * scale_k
    v = torch.randn(B, Hkv, N, d, generator=g)
    return [x.to(dtype).to(DEV) for x in (q, k, v)]


# ------------------------------------------------------------------ top-k --

def _topk_cases():
    rng = np.random.default_rng(0)
    cases = []
    # (32771: rows that do not start on a 16-byte boundary)
    for n, k in [(7, 3), (512, 32), (1000, 999), (4096, 512), (32768, 4096), (40000, 5000),
                 (131072, 8192), (32771, 4000)]:
        rows = 6
        x = rng.standard_normal((rows, n)).astype(np.float32)
        x[1] = np.round(x[1] * 2) / 2                # heavy ties
        x[2, ::3] = -0.0
        x[2, 1::3] = 0.0
        x[3, rng.random(n) < 0.2] = -np.inf
        x[4] = 1.0                                   # all equal: candidate overflow path
        cases.append((x, k))
    return cases


@pytest.mark.parametrize("case", range(8))
def test_topk_bit_exact_on_identical_scores(K, case):
    x, k = _topk_cases()[case]
    got = K.topk(torch.from_numpy(x).to(DEV), k).cpu().numpy()
    for r in range(x.shape[0]):
        assert got[r].tolist() == topk_indices(x[r], k).tolist(), (case, r)


def test_topk_long_row_fallbacks(K):
    """Long rows whose sample bracket cannot settle the k-th key: an 8192-key
    run set to the expected k-th value (its warps' candidate lists overflow),
    heavy keys placed only where the sample never looks (the k-th key lies
    above the bracket), few distinct values, and a NaN (reported as bad
    input). k = 1 and k = n rows ride along; every row must still follow the
    rule exactly."""
    rng = np.random.default_rng(23)
    n = 65536
    x = rng.standard_normal((5, n)).astype(np.float32)
    k = 4096
    # row 0: one 8192-key segment set to the expected k-th value (all candidates)
    kth = np.sort(x[0])[::-1][k - 1]
    x[0, 8192:16384] = kth
    # row 1: k + 100 heavy keys between the sample's runs (runs of 32 keys
    # start at multiples of (n - 32) / (runs - 1); keys 40..479 after each run
    # start are never sampled)
    runs = max(2048, min(8192, n // 16)) // 32
    step = (n - 32) / (runs - 1)
    starts = np.floor(np.arange(runs) * step).astype(np.int64)
    heavy = (starts[:, None] + np.arange(40, 480)[None, :]).ravel()
    heavy = heavy[heavy < n][: k + 100]
    x[1, heavy] = 50.0 + rng.random(heavy.size).astype(np.float32)
    # row 2: ties everywhere (a few distinct values)
    x[2] = np.round(x[2])
    got = K.topk(torch.from_numpy(x).to(DEV), k).cpu().numpy()
    for r in range(5):
        assert got[r].tolist() == topk_indices(x[r], k).tolist(), r
    for kk in (1, n):
        got = K.topk(torch.from_numpy(x[3:5].copy()).to(DEV), kk).cpu().numpy()
        for r in range(2):
            assert got[r].tolist() == topk_indices(x[3 + r], kk).tolist(), (kk, r)
    ws = K.Workspace(DEV)
    xn = torch.from_numpy(x[3:5].copy()).to(DEV)
    xn[1, 40000] = float("nan")
    K.topk(xn, k, ws=ws)
    assert ws.device_error() == K.BAD_INPUT
    got = K.topk(torch.from_numpy(x[3:5].copy()).to(DEV), k, ws=ws).cpu().numpy()
    assert ws.device_error() == K.OK
    assert got[0].tolist() == topk_indices(x[3], k).tolist()


def test_topk_many_short_rows_bit_exact(K):
    """1100 rows of 6000 keys take the 256-thread CTAs (the launch shape of the
    prefill tile rows); every row pattern of the cases above recurs across them,
    including the exact fallback (heavy ties, all equal)."""
    rng = np.random.default_rng(11)
    rows, n, k = 1100, 6000, 700
    x = rng.standard_normal((rows, n)).astype(np.float32)
    for r in range(rows):
        kind = r % 6
        if kind == 1:
            x[r] = np.round(x[r] * 2) / 2
        elif kind == 2:
            x[r, ::3] = -0.0
            x[r, 1::3] = 0.0
        elif kind == 3:
            x[r, rng.random(n) < 0.2] = -np.inf
        elif kind == 4:
            x[r] = 1.0
    got = K.topk(torch.from_numpy(x).to(DEV), k).cpu().numpy()
    for r in range(rows):
        assert got[r].tolist() == topk_indices(x[r], k).tolist(), r


def test_topk_nan_reported(K):
    ws = K.Workspace(DEV)
    x = torch.randn(3, 1000, device=DEV)
    x[1, 17] = float("nan")
    K.topk(x, 10, ws=ws)
    assert ws.device_error() == K.BAD_INPUT
    K.topk(torch.randn(3, 1000, device=DEV), 10, ws=ws)
    assert ws.device_error() == K.OK


# ------------------------------------------------------------ anchor/dense --

SHAPES = [  # B, Hq, Hkv, N, d, dtype
    (1, 4, 2, 512, 64, torch.float32),
    (1, 4, 2, 512, 64, torch.bfloat16),
    (2, 8, 8, 1000, 128, torch.bfloat16),     # G = 1, ragged N
    (2, 16, 2, 4097, 64, torch.bfloat16),     # G = 8, ragged tail over many tiles
    (3, 8, 2, 3000, 128, torch.bfloat16),     # G = 4
    (1, 4, 2, 70, 128, torch.bfloat16),       # shorter than one split
]


@pytest.mark.parametrize("shape", SHAPES)
def test_anchor_decode_matches_oracle(K, shape):
    B, Hq, Hkv, N, d, dt = shape
    q, k, v = _rand_layer(B, Hq, Hkv, N, d, dt, seed=N + Hq)
    topk = max(1, N // 8)
    out, idx, scores = K.anchor_decode(q, k, v, topk, return_scores=True)
    o_ref, _, s_ref = A.anchor_decode(f64(q), f64(k), f64(v), topk)
    tight = dt == torch.float32
    check_out(out, o_ref, *( (1e-4, 1e-5) if tight else (2e-2, 2e-3)))
    check_out(scores, s_ref, 1e-3, 1e-4, what="scores")
    got = idx.cpu().numpy()
    sc = scores.cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            check_index_set(got[b, h], s_ref[b, h], topk)
            # bit-exact against the oracle rule on the kernel's own fp32 scores
            assert got[b, h].tolist() == topk_indices(sc[b, h], topk).tolist()


@pytest.mark.parametrize("shape", SHAPES)
def test_dense_decode_matches_oracle_and_anchor(K, shape):
    B, Hq, Hkv, N, d, dt = shape
    q, k, v = _rand_layer(B, Hq, Hkv, N, d, dt, seed=3 * N + Hq)
    out = K.dense_decode(q, k, v)
    o_ref, _ = A.dense_decode(f64(q), f64(k), f64(v))
    check_out(out, o_ref, *((1e-4, 1e-5) if dt == torch.float32 else (2e-2, 2e-3)))
    out_a, _ = K.anchor_decode(q, k, v, max(1, N // 8))
    assert torch.equal(out, out_a)


def test_permuted_group_map(K):
    gm = [1, 0, 3, 2, 0, 1, 2, 3]
    q, k, v = _rand_layer(2, 8, 4, 777, 128, torch.bfloat16, seed=5)
    out, idx, scores = K.anchor_decode(q, k, v, 50, group_map=gm, return_scores=True)
    o_ref, idx_ref, s_ref = A.anchor_decode(f64(q), f64(k), f64(v), 50, gm)
    check_out(out, o_ref)
    got = idx.cpu().numpy()
    for b in range(2):
        for h in range(8):
            check_index_set(got[b, h], s_ref[b, h], 50)
    # the reuse kernel on the oracle's sets, against the oracle on the same sets
    out_r = K.reuse_decode(q, k, v, _dev_idx(idx_ref), group_map=gm)
    check_out(out_r, A.sparse_decode(f64(q), f64(k), f64(v), idx_ref, gm))


# ------------------------------------------------------------------- reuse --

@pytest.mark.parametrize("shape", SHAPES)
def test_reuse_decode_matches_oracle(K, shape):
    B, Hq, Hkv, N, d, dt = shape
    q, k, v = _rand_layer(B, Hq, Hkv, N, d, dt, seed=7 * N + Hq)
    topk = max(1, N // 8)
    _, idx_ref, _ = A.anchor_decode(f64(q), f64(k), f64(v), topk)   # the oracle's sets
    q2, k2, v2 = _rand_layer(B, Hq, Hkv, N, d, dt, seed=11 * N + Hq)
    out = K.reuse_decode(q2, k2, v2, _dev_idx(idx_ref))
    o_ref = A.sparse_decode(f64(q2), f64(k2), f64(v2), idx_ref)
    check_out(out, o_ref, *((1e-4, 1e-5) if dt == torch.float32 else (2e-2, 2e-3)))


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_reuse_with_all_keys_equals_dense(K, dt):
    q, k, v = _rand_layer(2, 8, 2, 640, 128 if dt == torch.bfloat16 else 64, dt, seed=9)
    N = k.shape[2]
    idx = torch.arange(N, dtype=torch.int32, device=DEV).expand(2, 8, N).contiguous()
    out_r = K.reuse_decode(q, k, v, idx)
    out_d = K.dense_decode(q, k, v)
    tol = 1e-5 if dt == torch.float32 else 1e-2
    assert (out_r.float() - out_d.float()).abs().max().item() <= tol


def test_reuse_poison_unselected_rows(K):
    B, Hq, Hkv, N, d = 2, 8, 2, 2048, 128
    q, k, v = _rand_layer(B, Hq, Hkv, N, d, torch.bfloat16, seed=13)
    _, idx = K.anchor_decode(q, k, v, 200)
    out = K.reuse_decode(q, k, v, idx)
    used = torch.zeros(B, Hkv, N, dtype=torch.bool, device=DEV)
    gm = default_gmap(Hq, Hkv)
    for h in range(Hq):
        used[:, gm[h]].scatter_(1, idx[:, h].long(), True)
    kp, vp = k.clone(), v.clone()
    kp[~used] = float("nan")
    vp[~used] = float("nan")
    out_p = K.reuse_decode(q, kp, vp, idx)
    assert torch.equal(out, out_p)
    # a selected row does change the output
    j = int(idx[0, 0, 0])
    vp2 = v.clone()
    vp2[0, 0, j] += 4.0
    assert not torch.equal(K.reuse_decode(q, k, vp2, idx)[0, 0], out[0, 0])


def test_reuse_bad_index_reported(K):
    ws = K.Workspace(DEV)
    q, k, v = _rand_layer(1, 4, 2, 256, 64, torch.bfloat16, seed=1)
    idx = torch.arange(16, dtype=torch.int32, device=DEV).expand(1, 4, 16).contiguous()
    idx[0, 1, 3] = 999
    K.reuse_decode(q, k, v, idx, ws=ws)
    assert ws.device_error() == K.BAD_INPUT


# ------------------------------------------------------------------- stack --

PLAN_SHAPES = [  # B, Hq, Hkv, N, d, k
    (2, 8, 2, 40000, 128, 1000),   # G = 4, many key-range chunks, a ragged last one
    (1, 16, 2, 5000, 64, 5000),    # G = 8, k = N: every key selected
    (3, 4, 4, 3001, 128, 7),       # G = 1, tiny k, ragged N
]


@pytest.mark.parametrize("shape", PLAN_SHAPES)
def test_stack_bitmap_plan_matches_layer_calls(K, shape):
    """In a bf16 per-head stack the reuse layers' union plan is built from the
    anchor Top-k's selection bitmaps; the single reuse call builds it from the
    index sets it is given. Both plans, and so the outputs, must be identical."""
    B, Hq, Hkv, N, d, k = shape
    layers = [_rand_layer(B, Hq, Hkv, N, d, torch.bfloat16, seed=N + 3 * l) for l in range(3)]
    qs, ks, vs = ([lay[i] for lay in layers] for i in range(3))
    outs, idx_buf = K.run_stack(K.DECODE, qs, ks, vs, k, [0])
    o0, i0 = K.anchor_decode(qs[0], ks[0], vs[0], k)
    o1 = K.reuse_decode(qs[1], ks[1], vs[1], i0)
    o2 = K.reuse_decode(qs[2], ks[2], vs[2], i0)
    assert torch.equal(idx_buf, i0)
    for a, b in zip(outs, [o0, o1, o2]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_stack_matches_layer_calls_and_oracle(K, dtype):
    w = configs.TINY_DECODE.with_(dtype=dtype, n_layers=5, anchors=(1, 3))
    qs, ks, vs = make_layers(w)
    dq, dk, dv = ([x.to(DEV) for x in xs] for xs in (qs, ks, vs))
    outs, idx_buf = K.run_stack(K.DECODE, dq, dk, dv, w.topk, list(w.anchors))
    # layer by layer through the single-layer entry points
    o0 = K.dense_decode(dq[0], dk[0], dv[0])
    o1, i1 = K.anchor_decode(dq[1], dk[1], dv[1], w.topk)
    o2 = K.reuse_decode(dq[2], dk[2], dv[2], i1)
    o3, i3 = K.anchor_decode(dq[3], dk[3], dv[3], w.topk)
    o4 = K.reuse_decode(dq[4], dk[4], dv[4], i3)
    for a, b in zip(outs, [o0, o1, o2, o3, o4]):
        assert torch.equal(a, b)
    assert torch.equal(idx_buf, i3)
    # against the oracle stack, which selects its own float64 sets
    ref_outs, _, written = run_oracle_stack("decode", [(f64(a_), f64(b_), f64(c_))
                                                       for a_, b_, c_ in zip(qs, ks, vs)],
                                            w.topk, list(w.anchors))
    # (the two sides pick their sets independently, so near-tie keys may
    # differ between them; the output tolerance absorbs such a swap)
    for o, r in zip(outs, ref_outs):
        check_out(o, r)
    for layer in (1, 3):
        s_ref = A.decode_logits(f64(qs[layer]), f64(ks[layer]), A.default_group_map(
            w.n_q_heads, w.n_kv_heads), A.default_scale(w.head_dim))
        got = (i1 if layer == 1 else i3).cpu().numpy()
        for b in range(w.batch):
            for h in range(w.n_q_heads):
                check_index_set(got[b, h], s_ref[b, h], w.topk)


# -------------------------------------------------------- full-size samples --

@pytest.mark.parametrize("cfg", ["llama8b", "gptoss"])
def test_full_size_decode_sampled(K, cfg):
    """The 8B (B=8, N=32768, k=4096) and gpt-oss-20b-like (B=4, N=131072,
    k=8192, d=64) decode shapes through the stack call, on sampled (sequence,
    head) units including the first and last: the anchor output and set
    against the oracle's decode_unit, the Top-k bit-exact on the kernel's own
    fp32 logits, and the reuse output over the oracle's own set."""
    w = configs.LLAMA8B_DECODE_32K if cfg == "llama8b" else configs.GPTOSS_DECODE_128K
    w = w.with_(n_layers=2)
    qs, ks, vs = make_layers(w, device=DEV)
    outs, idx = K.run_stack(K.DECODE, qs, ks, vs, w.topk, [0])
    # the anchor entry point with the logits buffer gives the stack's sets
    _, idx_a, s_gpu = K.anchor_decode(qs[0], ks[0], vs[0], w.topk, return_scores=True)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_a)
    gm = default_gmap(w.n_q_heads, w.n_kv_heads)
    scale = 1.0 / np.sqrt(w.head_dim)
    rng = np.random.default_rng(1)
    units = [(0, 0), (w.batch - 1, w.n_q_heads - 1)] + \
        [(int(rng.integers(w.batch)), int(rng.integers(w.n_q_heads))) for _ in range(6)]
    idx_np = idx.cpu().numpy()
    for b, h in units:
        g = gm[h]
        # one sequence and KV head on the host, mapped to index 0
        q0, K0, V0 = (f64(x[b:b + 1, sl]) for x, sl in
                      ((qs[0], slice(h, h + 1)), (ks[0], slice(g, g + 1)), (vs[0], slice(g, g + 1))))
        o_ref, sel, s_ref = A.decode_unit(q0, K0, V0, 0, 0, w.topk, [0], scale)
        check_out(outs[0][b, h], o_ref, what=("anchor out", b, h))
        check_topk_exact(idx_np[b, h], s_gpu[b, h].cpu().numpy(), w.topk, what=("top-k", b, h))
        check_index_set(idx_np[b, h], s_ref, w.topk, what=("set", b, h))
        q1, K1, V1 = (f64(x[b:b + 1, sl]) for x, sl in
                      ((qs[1], slice(h, h + 1)), (ks[1], slice(g, g + 1)), (vs[1], slice(g, g + 1))))
        o1_ref = A.decode_unit(q1, K1, V1, 0, 0, w.topk, [0], scale, idx=sel)
        check_out(outs[1][b, h], o1_ref, what=("reuse out", b, h))


@pytest.mark.parametrize("shape", [(1, 64, 8, 131072, 64, 8192), (1, 32, 8, 65536, 128, 8192),
                                   (2, 8, 1, 200000, 64, 4096)])
def test_few_units_long_rows(K, shape):
    """Few (sequence, KV head) units over a long cache: the reuse kernel takes
    long key-range chunks (its split limit), the dense kernel long splits. The
    anchor layer against the oracle (output, bit-exact Top-k on its own
    logits, sets by the near-tie rule), the reuse layer on the oracle's sets."""
    B, Hq, Hkv, N, d, k = shape
    q, kk, v = _rand_layer(B, Hq, Hkv, N, d, torch.bfloat16, seed=N + d)
    out, idx, s_gpu = K.anchor_decode(q, kk, v, k, return_scores=True)
    o_ref, idx_ref, s_ref = A.anchor_decode(f64(q), f64(kk), f64(v), k)
    check_out(out, o_ref)
    got, s_np = idx.cpu().numpy(), s_gpu.cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            check_topk_exact(got[b, h], s_np[b, h], k, what=("top-k", b, h))
            check_index_set(got[b, h], s_ref[b, h], k, what=("set", b, h))
    q2, k2, v2 = _rand_layer(B, Hq, Hkv, N, d, torch.bfloat16, seed=N + d + 1)
    out_r = K.reuse_decode(q2, k2, v2, _dev_idx(idx_ref))
    check_out(out_r, A.sparse_decode(f64(q2), f64(k2), f64(v2), idx_ref))


FUSED_SHAPES = [  # B, Hq, Hkv, N, d, k
    (8, 32, 8, 32768, 128, 4096),     # the 8B decode shape
    (4, 64, 8, 131072, 64, 8192),     # the gpt-oss-20b-like long shape
    (3, 8, 2, 3000, 128, 100),        # ragged splits, small k
    (1, 16, 2, 1500, 64, 1400),       # short row: the sample is the whole row
    (2, 8, 8, 70000, 128, 1),         # G = 1, k = 1
]


@pytest.mark.parametrize("shape", FUSED_SHAPES)
def test_fused_anchor_equals_two_kernel_anchor(K, shape):
    """kascade_anchor_decode_fused ranks the same fp32 logits under the same
    rule as kascade_anchor_decode: its sets, logits and outputs are identical
    bit for bit, and its sets follow the oracle rule on those logits."""
    B, Hq, Hkv, N, d, k = shape
    q, kk, v = _rand_layer(B, Hq, Hkv, N, d, torch.bfloat16, seed=N + k)
    ws = K.Workspace(DEV)
    out_f, idx_f, s_f = K.anchor_decode(q, kk, v, k, return_scores=True, ws=ws, fused=True)
    out_d, idx_d, s_d = K.anchor_decode(q, kk, v, k, return_scores=True, ws=ws)
    assert ws.device_error() == K.OK
    assert torch.equal(idx_f, idx_d) and torch.equal(s_f, s_d) and torch.equal(out_f, out_d)
    got, s_np = idx_f.cpu().numpy(), s_f.cpu().numpy()
    rng = np.random.default_rng(k)
    for b, h in [(0, 0), (B - 1, Hq - 1), (int(rng.integers(B)), int(rng.integers(Hq)))]:
        check_topk_exact(got[b, h], s_np[b, h], k, what=("fused top-k", b, h))


def test_anchor_decode_repeatable(K):
    """Every decode path that streams K/V through the TMA stage ring gives the
    same output bit for bit on every call. A stage refilled by TMA while a
    consumer warp still read its last V columns (no proxy fence between the
    warp's ldmatrix reads and the refill) made about one long-shape fused
    anchor layer in sixteen differ in one split's last output dims."""
    B, Hq, Hkv, N, d, k = FUSED_SHAPES[1]
    q, kk, v = _rand_layer(B, Hq, Hkv, N, d, torch.bfloat16, seed=N + k)
    ws = K.Workspace(DEV)
    ref = K.dense_decode(q, kk, v, ws=ws).clone()
    bad = []
    for rep in range(24):
        for name, o in (("fused", K.anchor_decode(q, kk, v, k, ws=ws, fused=True)[0]),
                        ("two-kernel", K.anchor_decode(q, kk, v, k, ws=ws)[0]),
                        ("dense", K.dense_decode(q, kk, v, ws=ws))):
            if not torch.equal(o, ref):
                bad.append((rep, name, int((o != ref).sum())))
    assert ws.device_error() == K.OK
    assert not bad, bad


@pytest.mark.parametrize("kind", ["equal", "ties", "sampled_heavy", "nan"])
def test_fused_anchor_topk_fallbacks(K, kind):
    """The fused anchor decode selects from the candidate lists its attention kernel
    files against a sample bracket; rows where the bracket misses take the
    full selection over the spilled logits. Every case must still equal the
    selection rule on the kernel's own fp32 logits: all logits equal (the
    lists overflow), a few distinct logits (heavy ties), heavy keys planted
    only where the sample looks (fewer than k keys reach the bracket), and a
    NaN key row (reported as bad input)."""
    B, Hq, Hkv, N, d, k = 2, 8, 2, 32768, 128, 256
    q, kk, v = _rand_layer(B, Hq, Hkv, N, d, torch.bfloat16, seed=61)
    if kind == "equal":
        q = torch.zeros_like(q)
    elif kind == "ties":
        rows = kk[:, :, :3].clone()
        kk = rows[:, :, torch.arange(N, device=DEV) % 3].contiguous()
    elif kind == "sampled_heavy":
        # the sample takes 64 evenly spaced runs of 32 keys (about 520 apart):
        # 100 heavy keys at the starts of 20 runs fill its top ranks, so its
        # bracket sits above all but about 100 keys of the row
        pos = torch.tensor([int(i * (N - 32) / 63) + e for i in range(20) for e in range(5)],
                           device=DEV)
        qd = q.float() / q.float().norm(dim=-1, keepdim=True)
        for b in range(B):
            for g in range(Hkv):
                u = qd[b, 4 * g:4 * g + 4].sum(0)
                kk[b, g, pos] = (6.0 * u / u.norm()).to(kk.dtype)
    elif kind == "nan":
        kk[1, 0, 777] = float("nan")
    ws = K.Workspace(DEV)
    out, idx, s_gpu = K.anchor_decode(q, kk, v, k, return_scores=True, ws=ws, fused=True)
    if kind == "nan":
        assert ws.device_error() == K.BAD_INPUT
        return
    assert ws.device_error() == K.OK
    got, s_np = idx.cpu().numpy(), s_gpu.cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            check_topk_exact(got[b, h], s_np[b, h], k, what=(kind, b, h))
    if kind == "equal":
        assert (got == np.arange(k)).all()
    check_out(out, A.dense_decode(f64(q), f64(kk), f64(v))[0])


def test_workspace_shared_across_shapes_and_entry_points(K):
    """One workspace serves calls of different shapes and the overlap kernel;
    the split counters they rely on must survive every other call's writes."""
    ws = K.Workspace(DEV)
    shapes = [(8, 32, 8, 2048, 128), (2, 8, 2, 3000, 128), (4, 16, 2, 1500, 64)]
    layers = [_rand_layer(B, Hq, Hkv, N, d, torch.bfloat16, seed=40 + i)
              for i, (B, Hq, Hkv, N, d) in enumerate(shapes)]
    sets = torch.randint(0, 4096, (3, 16, 64), device=DEV, dtype=torch.int32)
    for rep in range(2):
        for (q, k, v) in layers:
            out = K.dense_decode(q, k, v, ws=ws)
            check_out(out, A.dense_decode(f64(q), f64(k), f64(v))[0])
            _, idx = K.anchor_decode(q, k, v, 64, ws=ws)
            _, idx_ref, s_ref = A.anchor_decode(f64(q), f64(k), f64(v), 64)
            got = idx.cpu().numpy()
            for b_ in range(got.shape[0]):
                for h_ in range(got.shape[1]):
                    check_index_set(got[b_, h_], s_ref[b_, h_], 64)
            out_r = K.reuse_decode(q, k, v, _dev_idx(idx_ref), ws=ws)
            check_out(out_r, A.sparse_decode(f64(q), f64(k), f64(v), idx_ref))
            K.layer_overlap(sets, 4096, ws=ws)
    assert ws.device_error() == K.OK


def test_bounded_wait_times_out_and_context_survives(K):
    """A device wait on a barrier nothing completes gives up after the wait
    limit, reports KASCADE_ERR_TIMEOUT, and the next launches run normally."""
    import time
    ws = K.Workspace(DEV)
    t0 = time.perf_counter()
    assert ws.check_wait_timeout() == K.TIMEOUT
    assert time.perf_counter() - t0 < 30.0
    assert ws.device_error() == K.OK          # the word was read and cleared
    q, k, v = _rand_layer(1, 4, 2, 256, 64, torch.bfloat16, seed=3)
    out = K.dense_decode(q, k, v, ws=ws)
    check_out(out, A.dense_decode(f64(q), f64(k), f64(v))[0])
    assert ws.device_error() == K.OK
