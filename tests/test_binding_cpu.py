"""The Python binding checks every tensor against the extents its descriptor
implies before handing the address to the library: the layouts the library
documents pass, and a wrong shape, dtype, device, layer count or a
non-contiguous tensor raises before any library call. No GPU: the library is
replaced by a recorder, and the accepted device type is pointed at the CPU
for the calls that must pass."""
import pytest
import torch

import __graft_entry__

BF = torch.bfloat16


@pytest.fixture(scope="module")
def K():
    __graft_entry__.build()
    from long_context_anchor_gb300 import kascade
    return kascade


class _Recorder:
    """Stands in for the shared library: sizes are small, every call succeeds."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append(name)
            if name.endswith("workspace_size"):
                return 4096
            if name == "kascade_status_string":
                return b"fake"
            return 0
        return fn


@pytest.fixture
def fake(K, monkeypatch):
    rec = _Recorder()
    monkeypatch.setattr(K, "_lib", rec)
    monkeypatch.setattr(K, "_stream", lambda stream=None: None)
    monkeypatch.setattr(K, "_DEVICE_TYPE", "cpu")
    return rec


def _decode(B=2, Hq=8, Hkv=2, N=300, d=64, dtype=BF):
    return (torch.zeros(B, Hq, d, dtype=dtype), torch.zeros(B, Hkv, N, d, dtype=dtype),
            torch.zeros(B, Hkv, N, d, dtype=dtype))


def _prefill(B=1, Hq=4, Hkv=2, N=300, d=128):
    return (torch.zeros(B, Hq, N, d, dtype=BF), torch.zeros(B, Hkv, N, d, dtype=BF),
            torch.zeros(B, Hkv, N, d, dtype=BF))


def test_documented_layouts_pass(K, fake):
    ws = K.Workspace("cpu")
    q, k, v = _decode()
    assert K.dense_decode(q, k, v, ws=ws).shape == q.shape
    out, idx = K.anchor_decode(q, k, v, 32, ws=ws)
    assert idx.shape == (2, 8, 32) and idx.dtype == torch.int32
    out, idx, s = K.anchor_decode(q, k, v, 32, return_scores=True, pooled=True, ws=ws)
    assert idx.shape == (2, 2, 32) and s.shape == (2, 2, 300)
    K.reuse_decode(q, k, v, torch.zeros(2, 8, 32, dtype=torch.int32), ws=ws)
    K.reuse_decode(q, k, v, torch.zeros(2, 2, 32, dtype=torch.int32), pooled=True, ws=ws)
    K.anchor_decode(q, k, v, 32, out=torch.empty_like(q),
                    idx=torch.empty(2, 8, 32, dtype=torch.int32), ws=ws)
    assert K.topk(torch.zeros(5, 100), 7, ws=ws).shape == (5, 7)
    assert K.topk(torch.zeros(0, 100), 7, ws=ws).shape == (0, 7)
    q, k, v = _prefill()
    K.dense_prefill(q, k, v, ws=ws)
    out, idx = K.anchor_prefill(q, k, v, 40, ws=ws)
    assert idx.shape == (1, 4, 3, 40)
    out, idx, wts = K.anchor_prefill(q, k, v, 40, ws=ws, return_weights=True)
    # packed tile rows: L_0 + L_1 + L_2 = 128 + 256 + 300
    assert wts.shape == (1, 4, 684) and K.packed_tile_len(300) == 684
    assert [K.packed_tile_offset(t) for t in range(3)] == [0, 128, 384]
    _, _, wts = K.anchor_prefill(q, k, v, 40, ws=ws, return_weights=True, pooled=True)
    assert wts.shape == (1, 2, 684)
    K.reuse_prefill(q, k, v, torch.zeros(1, 2, 3, 40, dtype=torch.int32), pooled=True, ws=ws)
    qs, ks, vs = [list(t) for t in (q.expand(3, *q.shape).contiguous(),
                                    k.expand(3, *k.shape).contiguous(),
                                    v.expand(3, *v.shape).contiguous())]
    outs, ib = K.run_stack(K.PREFILL, qs, ks, vs, 40, [0], ws=ws)
    assert ib.shape == (1, 4, 3, 40) and len(outs) == 3
    qd, kd, vd = _decode()
    stack = [list(t.expand(4, *t.shape).contiguous()) for t in (qd, kd, vd)]
    K.run_stack(K.DECODE, *stack, 16, [0, 2], outs=[torch.empty_like(qd) for _ in range(4)],
                idx_buf=torch.empty(2, 2, 16, dtype=torch.int32), pooled=True, ws=ws)
    sim, sets = K.calibrate(*stack, 16, ws=ws)
    assert sets.shape == (4, 16, 16)
    K.layer_overlap(torch.zeros(4, 16, 16, dtype=torch.int32), 300, ws=ws)
    assert "kascade_run_stack" in fake.calls and "kascade_calibrate" in fake.calls


def _compute_calls(rec):
    return [c for c in rec.calls if not c.endswith("workspace_size") and c != "kascade_workspace_init"
            and c != "kascade_status_string"]


@pytest.mark.parametrize("case", range(12))
def test_mismatched_tensors_raise_before_the_library(K, fake, case):
    q, k, v = _decode()
    i32 = torch.int32
    with pytest.raises((ValueError, TypeError)):
        if case == 0:
            K.dense_decode(q, k, v[:, :, :299].contiguous())        # v shorter than k
        elif case == 1:
            K.dense_decode(q, k.float(), v)                         # k dtype differs from q
        elif case == 2:
            K.dense_decode(q, k, v, out=torch.empty(2, 8, 32, dtype=BF))
        elif case == 3:
            K.reuse_decode(q, k, v, torch.zeros(2, 8, 32, dtype=torch.int64))
        elif case == 4:
            K.reuse_decode(q, k, v, torch.zeros(2, 2, 32, dtype=i32))   # per-head mode, Hkv rows
        elif case == 5:
            K.anchor_decode(q, k, v, 32, idx=torch.empty(2, 8, 31, dtype=i32))
        elif case == 6:
            K.dense_decode(q, k.transpose(2, 3), v)                 # wrong layout
        elif case == 7:
            K.topk(torch.zeros(5, 100, dtype=torch.float64), 7)
        elif case == 8:
            qp, kp, vp = _prefill()
            K.reuse_prefill(qp, kp, vp, torch.zeros(1, 4, 2, 40, dtype=i32))   # nT = 3
        elif case == 9:
            qp, kp, vp = _prefill()
            K.run_stack(K.PREFILL, [qp, qp], [kp], [vp, vp], 40, [0])
        elif case == 10:
            qp, kp, vp = _prefill()
            K.run_stack(K.PREFILL, [qp, qp[:, :, :200].contiguous()], [kp, kp], [vp, vp], 40, [0])
        else:
            base = torch.zeros(2, 8, 128, dtype=BF)
            K.dense_decode(base[:, :, ::2], k, v)                   # not contiguous
    assert _compute_calls(fake) == []


def test_host_tensors_are_refused(K, monkeypatch):
    rec = _Recorder()
    monkeypatch.setattr(K, "_lib", rec)
    q, k, v = _decode()
    with pytest.raises(ValueError, match="CUDA"):
        K.dense_decode(q, k, v)
    with pytest.raises(ValueError, match="CUDA"):
        K.topk(torch.zeros(3, 10), 2)
    assert rec.calls == []


def test_kascade_attention_dispatches_on_query_rank(K, fake, monkeypatch):
    seen = []
    real = K.run_stack

    def spy(mode, *a, **kw):
        seen.append(mode)
        return real(mode, *a, **kw)

    monkeypatch.setattr(K, "run_stack", spy)
    ws = K.Workspace("cpu")
    qd, kd, vd = _decode()
    outs = K.kascade_attention([qd, qd], [kd, kd], [vd, vd], 16, [1], ws=ws)
    assert len(outs) == 2 and outs[0].shape == qd.shape
    qp, kp, vp = _prefill()
    K.kascade_attention([qp], [kp], [vp], 40, (0,), ws=ws)
    assert seen == [K.DECODE, K.PREFILL]
    with pytest.raises(ValueError):
        K.kascade_attention([], [], [], 16, [0])

