"""Python binding of libkascade (include/kascade.h).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels. PyTorch supplies device memory (outputs, the
workspace) and the current CUDA stream. Importing this module loads
``libkascade.so`` from this package directory and raises if it is missing;
there is no fallback.
"""
import ctypes
import math
import os
from typing import List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkascade.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libkascade.so is not built; run python -m long_context_anchor_gb300.build "
                      "(or __graft_entry__.build())")
_lib = ctypes.CDLL(LIB_PATH)

OK, INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA, BAD_INPUT, TIMEOUT = range(7)
F32, BF16 = 0, 1
DECODE, PREFILL = 0, 1
PER_QHEAD, PER_KVHEAD = 0, 1     # kascade_index_mode: per query head, or GQA-pooled
TILE = 128


class Desc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_len", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("scale", ctypes.c_float), ("group_map", ctypes.POINTER(ctypes.c_int32)),
                ("index_mode", ctypes.c_int32)]


_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_DP = ctypes.POINTER(Desc)
_SIGS = {
    "kascade_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kascade_workspace_size": (_sz, [_DP, _i32, _i32]),
    "kascade_workspace_init": (ctypes.c_int, [_vp, _sz, _vp]),
    "kascade_device_error": (ctypes.c_int, [_vp, _vp]),
    "kascade_check_wait_timeout": (ctypes.c_int, [_vp, _sz, _vp]),
    "kascade_dense_decode": (ctypes.c_int, [_DP, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "kascade_anchor_decode": (ctypes.c_int, [_DP, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "kascade_anchor_decode_fused": (ctypes.c_int, [_DP, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp,
                                                   _sz, _vp]),
    "kascade_reuse_decode": (ctypes.c_int, [_DP, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp]),
    "kascade_topk": (ctypes.c_int, [_vp, _i32, _i32, _i32, _vp, _vp, _sz, _vp]),
    "kascade_dense_decode_noalloc": (ctypes.c_int, [_DP, _vp, _vp, _vp, _vp, _vp]),
    "kascade_noalloc_device_error": (ctypes.c_int, [_vp]),
    "kascade_anchor_decode_shard": (ctypes.c_int, [_DP, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp,
                                                   _vp, _vp, _sz, _vp]),
    "kascade_merge_workspace_size": (_sz, [_DP, _i32, _i32]),
    "kascade_merge_decode_shards": (ctypes.c_int, [_DP, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _vp,
                                                   _vp, _sz, _vp]),
    "kascade_dense_prefill": (ctypes.c_int, [_DP, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "kascade_anchor_prefill": (ctypes.c_int, [_DP, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _sz,
                                              _vp]),
    "kascade_reuse_prefill": (ctypes.c_int, [_DP, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp]),
    "kascade_run_stack": (ctypes.c_int, [_DP, _i32, _i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                         ctypes.POINTER(_vp), _i32, ctypes.POINTER(_i32), _i32,
                                         ctypes.POINTER(_vp), _vp, _vp, _sz, _vp]),
    "kascade_run_stack_profiled": (ctypes.c_int, [_DP, _i32, _i32, ctypes.POINTER(_vp),
                                                  ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i32,
                                                  ctypes.POINTER(_i32), _i32, ctypes.POINTER(_vp),
                                                  _vp, _vp, _sz, _vp, ctypes.POINTER(_vp)]),
    "kascade_overlap_workspace_size": (_sz, [_i32, _i32, _i32]),
    "kascade_calibrate_workspace_size": (_sz, [_DP, _i32, _i32]),
    "kascade_calibrate": (ctypes.c_int, [_DP, _i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                         ctypes.POINTER(_vp), _i32, ctypes.POINTER(_vp), _vp,
                                         ctypes.POINTER(ctypes.c_double), _vp, _sz, _vp]),
    "kascade_calibrate_recall_workspace_size": (_sz, [_DP, _i32, _i32]),
    "kascade_calibrate_recall": (ctypes.c_int, [_DP, _i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                                ctypes.POINTER(_vp), _i32, ctypes.POINTER(_vp), _vp,
                                                ctypes.POINTER(ctypes.c_double), _vp, _sz, _vp]),
    "kascade_layer_overlap": (ctypes.c_int, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _sz, _vp]),
    "kascade_schedule_anchors": (ctypes.c_int, [ctypes.POINTER(ctypes.c_double), _i32, _i32,
                                                ctypes.POINTER(_i32), ctypes.POINTER(ctypes.c_double)]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


class KascadeError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))
        self.status = status


def status_string(s: int) -> str:
    return _lib.kascade_status_string(int(s)).decode()


def _check(status: int, where: str):
    if status != OK:
        raise KascadeError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_desc(batch, n_q_heads, n_kv_heads, head_dim, kv_len, dtype, scale=0.0,
              group_map: Optional[Sequence[int]] = None, pooled: bool = False):
    d = Desc(batch, n_q_heads, n_kv_heads, head_dim, kv_len, dtype,
             float(scale or 0.0), None, PER_KVHEAD if pooled else PER_QHEAD)
    keep = None
    if group_map is not None:
        keep = (ctypes.c_int32 * n_q_heads)(*[int(x) for x in group_map])
        d.group_map = ctypes.cast(keep, ctypes.POINTER(ctypes.c_int32))
    d._keep = keep      # keep the host array alive with the descriptor
    return d


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError("q/k/v must be bfloat16 or float32")


def decode_desc(q, k, group_map=None, scale=None, pooled=False):
    B, Hq, d = q.shape
    _, Hkv, N, _ = k.shape
    return make_desc(B, Hq, Hkv, d, N, _dtype_code(q), scale or 0.0, group_map, pooled)


def prefill_desc(q, k, group_map=None, scale=None, pooled=False):
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    return make_desc(B, Hq, Hkv, d, N, _dtype_code(q), scale or 0.0, group_map, pooled)


def workspace_size(desc, topk: int, mode: int) -> int:
    n = _lib.kascade_workspace_size(ctypes.byref(desc), int(topk), int(mode))
    if n == 0:
        raise KascadeError(INVALID_ARG, "kascade_workspace_size")
    return n


class Workspace:
    """Caller-owned device workspace (torch memory), zeroed once when (re)allocated."""

    def __init__(self, device=None):
        self.device = torch.device(device if device is not None else "cuda")
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int, stream=None) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
            _check(_lib.kascade_workspace_init(_ptr(self.buf), self.buf.numel(), _stream(stream)),
                   "kascade_workspace_init")
        return self.buf

    def check_wait_timeout(self, stream=None) -> int:
        """Run one device wait that can only time out; returns the device error status."""
        buf = self.get(256, stream)
        _check(_lib.kascade_check_wait_timeout(_ptr(buf), buf.numel(), _stream(stream)),
               "kascade_check_wait_timeout")
        return self.device_error(stream)

    def device_error(self, stream=None) -> int:
        """Synchronise and read/clear the device error word (an int status)."""
        if self.buf is None:
            return OK
        return _lib.kascade_device_error(_ptr(self.buf), _stream(stream))


_default_ws = {}


def default_workspace(device) -> Workspace:
    dev = torch.device(device)
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    if key not in _default_ws:
        _default_ws[key] = Workspace(torch.device("cuda", key))
    return _default_ws[key]


def _ws(ws, device, nbytes, stream):
    ws = ws if ws is not None else default_workspace(device)
    buf = ws.get(nbytes, stream)
    return ws, buf


# The library reads and writes raw device pointers with the extents the
# descriptor implies, so every tensor is checked against those extents here,
# before its address is handed over: a wrong shape, dtype or device would
# otherwise become an out-of-bounds access on the GPU.

def _expect(t, name, shape, dtype):
    """Shape, dtype and contiguity of one tensor (no device check)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s: expected a torch.Tensor" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s: shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if t.dtype != dtype:
        raise TypeError("%s: dtype %s, expected %s" % (name, t.dtype, dtype))
    if not t.is_contiguous():
        raise ValueError("%s: must be contiguous" % name)


_DEVICE_TYPE = "cuda"   # the only device type whose addresses the library takes


def _same_cuda_device(named):
    """All tensors on one CUDA device; returns it."""
    dev = named[0][1].device
    if dev.type != _DEVICE_TYPE:
        raise ValueError("%s: on %s; the library takes CUDA device tensors" % (named[0][0], dev))
    for name, t in named[1:]:
        if t.device != dev:
            raise ValueError("%s: on %s, expected %s" % (name, t.device, dev))
    return dev


def _attn_inputs(q, k, v, prefill: bool):
    """Validated (B, Hq, Hkv, N, d) of one layer's q, k, v.

    decode: q [B,Hq,d], k/v [B,Hkv,N,d]; prefill: q [B,Hq,N,d], k/v [B,Hkv,N,d].
    k and v take q's dtype (bf16 or fp32)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s: expected a torch.Tensor" % name)
    if q.dim() != (4 if prefill else 3) or k.dim() != 4:
        raise ValueError("q must be %s and k, v [B,Hkv,N,d]; got q %s, k %s"
                         % ("[B,Hq,N,d]" if prefill else "[B,Hq,d]", tuple(q.shape),
                            tuple(k.shape)))
    _dtype_code(q)
    B, Hq, d = q.shape[0], q.shape[1], q.shape[-1]
    Hkv, N = k.shape[1], k.shape[2]
    if prefill and q.shape[2] != N:
        raise ValueError("q: %d rows, k: %d keys; prefill needs both equal" % (q.shape[2], N))
    _expect(q, "q", q.shape, q.dtype)
    _expect(k, "k", (B, Hkv, N, d), q.dtype)
    _expect(v, "v", (B, Hkv, N, d), q.dtype)
    return B, Hq, Hkv, N, d


def _all_like(ts, name, shape, dtype, dev):
    """Every tensor of a per-layer list has this shape, dtype and device and is
    contiguous (one fast pass; the first mismatch gets a detailed error)."""
    for l, t in enumerate(ts):
        if not (isinstance(t, torch.Tensor) and t.shape == shape and t.dtype == dtype
                and t.device == dev and t.is_contiguous()):
            _expect(t, "%s[%d]" % (name, l), shape, dtype)
            raise ValueError("%s[%d]: on %s, expected %s" % (name, l, t.device, dev))


def _layers(qs, ks, vs, prefill: bool):
    """Validated stack inputs: every layer has layer 0's shapes, dtype and
    device; returns (B, Hq, Hkv, N, d) and the device."""
    L = len(qs)
    if L < 1 or len(ks) != L or len(vs) != L:
        raise ValueError("qs, ks, vs: one tensor per layer each (got %d, %d, %d)"
                         % (len(qs), len(ks), len(vs)))
    sizes = _attn_inputs(qs[0], ks[0], vs[0], prefill)
    dev = _same_cuda_device([("qs[0]", qs[0]), ("ks[0]", ks[0]), ("vs[0]", vs[0])])
    _all_like(qs, "qs", qs[0].shape, qs[0].dtype, dev)
    _all_like(ks, "ks", ks[0].shape, qs[0].dtype, dev)
    _all_like(vs, "vs", ks[0].shape, qs[0].dtype, dev)
    return sizes, dev


# ------------------------------------------------------------------ decode --

def dense_decode(q, k, v, group_map=None, scale=None, out=None, ws=None, stream=None):
    """Exact decode attention: q [B,Hq,d], k/v [B,Hkv,N,d] -> out [B,Hq,d]."""
    _attn_inputs(q, k, v, prefill=False)
    if out is not None:
        _expect(out, "out", q.shape, q.dtype)
    _same_cuda_device([("q", q), ("k", k), ("v", v)] + ([("out", out)] if out is not None else []))
    desc = decode_desc(q, k, group_map, scale)
    out = torch.empty_like(q) if out is None else out
    ws, buf = _ws(ws, q.device, workspace_size(desc, 1, DECODE), stream)
    _check(_lib.kascade_dense_decode(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                     _ptr(buf), buf.numel(), _stream(stream)), "kascade_dense_decode")
    return out


def anchor_decode(q, k, v, topk, group_map=None, scale=None, return_scores=False, out=None,
                  idx=None, ws=None, stream=None, pooled=False, fused=False):
    """Anchor layer: (out [B,Hq,d], idx [B,H,topk] int32[, scores [B,H,N] fp32]).

    H = Hq: per-head sets, scores = the scaled logits. pooled: H = Hkv, one
    set per KV head, scores = the group sums of the softmax weights. fused:
    the Top-k fused into the attention kernel (kascade_anchor_decode_fused;
    bf16, per-head sets; the same results)."""
    B, Hq, Hkv, N, _ = _attn_inputs(q, k, v, prefill=False)
    H = Hkv if pooled else Hq
    extra = []
    if out is not None:
        _expect(out, "out", q.shape, q.dtype)
        extra.append(("out", out))
    if idx is not None:
        _expect(idx, "idx", (B, H, topk), torch.int32)
        extra.append(("idx", idx))
    _same_cuda_device([("q", q), ("k", k), ("v", v)] + extra)
    desc = decode_desc(q, k, group_map, scale, pooled)
    out = torch.empty_like(q) if out is None else out
    idx = torch.empty(B, H, topk, dtype=torch.int32, device=q.device) if idx is None else idx
    scores = torch.empty(B, H, N, dtype=torch.float32, device=q.device) if return_scores else None
    ws, buf = _ws(ws, q.device, workspace_size(desc, topk, DECODE), stream)
    fn, name = ((_lib.kascade_anchor_decode_fused, "kascade_anchor_decode_fused") if fused
                else (_lib.kascade_anchor_decode, "kascade_anchor_decode"))
    _check(fn(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), int(topk), _ptr(out), _ptr(idx),
              _ptr(scores), _ptr(buf), buf.numel(), _stream(stream)), name)
    return (out, idx, scores) if return_scores else (out, idx)


def reuse_decode(q, k, v, idx, group_map=None, scale=None, out=None, ws=None, stream=None,
                 pooled=False):
    """Reuse layer over saved sets idx [B,Hq,topk] (pooled: [B,Hkv,topk]; int32, ascending)."""
    B, Hq, Hkv, _, _ = _attn_inputs(q, k, v, prefill=False)
    if not isinstance(idx, torch.Tensor) or idx.dim() != 3:
        raise ValueError("idx: expected an int32 tensor [B,H,topk]")
    topk = idx.shape[-1]
    _expect(idx, "idx", (B, Hkv if pooled else Hq, topk), torch.int32)
    extra = [("idx", idx)]
    if out is not None:
        _expect(out, "out", q.shape, q.dtype)
        extra.append(("out", out))
    _same_cuda_device([("q", q), ("k", k), ("v", v)] + extra)
    desc = decode_desc(q, k, group_map, scale, pooled)
    out = torch.empty_like(q) if out is None else out
    ws, buf = _ws(ws, q.device, workspace_size(desc, topk, DECODE), stream)
    _check(_lib.kascade_reuse_decode(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), int(topk),
                                     _ptr(idx), _ptr(out), _ptr(buf), buf.numel(), _stream(stream)),
           "kascade_reuse_decode")
    return out


def anchor_decode_shard(q, k, v, key_offset, topk, group_map=None, scale=None, ws=None,
                        stream=None):
    """One shard of a KV cache split along the key axis: k/v [B,Hkv,N_s,d] hold
    global positions key_offset .. key_offset + N_s - 1. Returns the shard's
    partials (out [B,Hq,d], lse [B,Hq] fp32, cand_idx [B,Hq,topk] int32 global
    positions ascending, cand_scores [B,Hq,topk] fp32 logits)."""
    B, Hq, _, N, _ = _attn_inputs(q, k, v, prefill=False)
    _same_cuda_device([("q", q), ("k", k), ("v", v)])
    if not (1 <= int(topk) <= N) or int(key_offset) < 0:
        raise ValueError("topk must lie in [1, N_s] and key_offset must be >= 0")
    desc = decode_desc(q, k, group_map, scale)
    out = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    cand_idx = torch.empty(B, Hq, topk, dtype=torch.int32, device=q.device)
    cand_scores = torch.empty(B, Hq, topk, dtype=torch.float32, device=q.device)
    ws, buf = _ws(ws, q.device, workspace_size(desc, topk, DECODE), stream)
    _check(_lib.kascade_anchor_decode_shard(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v),
                                            int(key_offset), int(topk), _ptr(out), _ptr(lse),
                                            _ptr(cand_idx), _ptr(cand_scores), _ptr(buf),
                                            buf.numel(), _stream(stream)),
           "kascade_anchor_decode_shard")
    return out, lse, cand_idx, cand_scores


def merge_decode_shards(outs, lses, cand_idx, cand_scores, n_kv_heads=None, kv_len=None,
                        ws=None, stream=None):
    """Merge S shards' partials stacked in key order: outs [S,B,Hq,d], lses
    [S,B,Hq] fp32, cand_idx [S,B,Hq,topk] int32, cand_scores [S,B,Hq,topk]
    fp32. Returns (out [B,Hq,d], idx [B,Hq,topk] ascending global positions).
    kv_len (the total keys, for the range check of the candidates) defaults
    to the largest candidate position + 1; n_kv_heads to Hq (the merge does
    not read K or V)."""
    if not isinstance(outs, torch.Tensor) or outs.dim() != 4:
        raise ValueError("outs: expected a tensor [S,B,Hq,d]")
    S, B, Hq, d = outs.shape
    if not isinstance(cand_idx, torch.Tensor) or cand_idx.dim() != 4:
        raise ValueError("cand_idx: expected an int32 tensor [S,B,Hq,topk]")
    topk = cand_idx.shape[-1]
    _expect(lses, "lses", (S, B, Hq), torch.float32)
    _expect(cand_idx, "cand_idx", (S, B, Hq, topk), torch.int32)
    _expect(cand_scores, "cand_scores", (S, B, Hq, topk), torch.float32)
    _expect(outs, "outs", (S, B, Hq, d), outs.dtype)
    _same_cuda_device([("outs", outs), ("lses", lses), ("cand_idx", cand_idx),
                       ("cand_scores", cand_scores)])
    if kv_len is None:
        kv_len = int(cand_idx.max().item()) + 1
    hkv = Hq if n_kv_heads is None else int(n_kv_heads)
    desc = make_desc(B, Hq, hkv, d, int(kv_len), _dtype_code(outs))
    out = torch.empty(B, Hq, d, dtype=outs.dtype, device=outs.device)
    idx = torch.empty(B, Hq, topk, dtype=torch.int32, device=outs.device)
    n = _lib.kascade_merge_workspace_size(ctypes.byref(desc), int(S), int(topk))
    if n == 0:
        raise KascadeError(INVALID_ARG, "kascade_merge_workspace_size")
    ws, buf = _ws(ws, outs.device, n, stream)
    _check(_lib.kascade_merge_decode_shards(ctypes.byref(desc), int(S), _ptr(outs), _ptr(lses),
                                            _ptr(cand_idx), _ptr(cand_scores), int(topk),
                                            _ptr(out), _ptr(idx), _ptr(buf), buf.numel(),
                                            _stream(stream)), "kascade_merge_decode_shards")
    return out, idx


def topk(scores, k, out=None, ws=None, stream=None):
    """Exact Top-k of fp32 rows [rows, n] -> int32 [rows, k] ascending."""
    if not isinstance(scores, torch.Tensor) or scores.dim() != 2:
        raise ValueError("scores: expected an fp32 tensor [rows, n]")
    rows, n = scores.shape
    _expect(scores, "scores", (rows, n), torch.float32)
    named = [("scores", scores)]
    if out is not None:
        _expect(out, "out", (rows, int(k)), torch.int32)
        named.append(("out", out))
    _same_cuda_device(named)
    out = torch.empty(rows, k, dtype=torch.int32, device=scores.device) if out is None else out
    ws, buf = _ws(ws, scores.device, 256, stream)
    _check(_lib.kascade_topk(_ptr(scores), rows, n, int(k), _ptr(out), _ptr(buf), buf.numel(),
                             _stream(stream)), "kascade_topk")
    return out


# ----------------------------------------------------------------- prefill --

def n_tiles(n: int) -> int:
    return (n + TILE - 1) // TILE


def dense_prefill(q, k, v, group_map=None, scale=None, out=None, ws=None, stream=None):
    """Causal exact attention: q [B,Hq,N,d], k/v [B,Hkv,N,d] (bf16)."""
    _attn_inputs(q, k, v, prefill=True)
    if out is not None:
        _expect(out, "out", q.shape, q.dtype)
    _same_cuda_device([("q", q), ("k", k), ("v", v)] + ([("out", out)] if out is not None else []))
    desc = prefill_desc(q, k, group_map, scale)
    out = torch.empty_like(q) if out is None else out
    ws, buf = _ws(ws, q.device, workspace_size(desc, 1, PREFILL), stream)
    _check(_lib.kascade_dense_prefill(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                      _ptr(buf), buf.numel(), _stream(stream)), "kascade_dense_prefill")
    return out


def packed_tile_len(n: int) -> int:
    """Length of one (sequence, head) row of packed tile weights: sum_t L_t."""
    nt = n_tiles(n)
    return 64 * (nt - 1) * nt + n


def packed_tile_offset(t: int) -> int:
    """Offset of tile t's weights in a packed row (64 t (t + 1))."""
    return 64 * t * (t + 1)


def anchor_prefill(q, k, v, topk, group_map=None, scale=None, out=None, idx=None, ws=None,
                   stream=None, pooled=False, return_weights=False):
    """Anchor layer, prefill: (out, idx [B,H,nT,topk] int32, -1 padded), H = Hq or,
    pooled, Hkv. With return_weights, also the fp32 tile weights the selection
    ranked, packed [B,H,packed_tile_len(N)] (tile t at packed_tile_offset(t),
    L_t = min(N, 128(t+1)) entries): (out, idx, weights)."""
    B, Hq, Hkv, N, _ = _attn_inputs(q, k, v, prefill=True)
    H = Hkv if pooled else Hq
    extra = []
    if out is not None:
        _expect(out, "out", q.shape, q.dtype)
        extra.append(("out", out))
    if idx is not None:
        _expect(idx, "idx", (B, H, n_tiles(N), topk), torch.int32)
        extra.append(("idx", idx))
    _same_cuda_device([("q", q), ("k", k), ("v", v)] + extra)
    desc = prefill_desc(q, k, group_map, scale, pooled)
    out = torch.empty_like(q) if out is None else out
    if idx is None:
        idx = torch.empty(B, H, n_tiles(N), topk, dtype=torch.int32, device=q.device)
    wts = (torch.empty(B, H, packed_tile_len(N), dtype=torch.float32, device=q.device)
           if return_weights else None)
    ws, buf = _ws(ws, q.device, workspace_size(desc, topk, PREFILL), stream)
    _check(_lib.kascade_anchor_prefill(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), int(topk),
                                       _ptr(out), _ptr(idx), _ptr(wts), _ptr(buf), buf.numel(),
                                       _stream(stream)), "kascade_anchor_prefill")
    return (out, idx, wts) if return_weights else (out, idx)


def reuse_prefill(q, k, v, idx, group_map=None, scale=None, out=None, ws=None, stream=None,
                  pooled=False):
    """Reuse layer, prefill, over saved tile sets idx [B,Hq,nT,topk] (pooled: [B,Hkv,nT,topk])."""
    B, Hq, Hkv, N, _ = _attn_inputs(q, k, v, prefill=True)
    if not isinstance(idx, torch.Tensor) or idx.dim() != 4:
        raise ValueError("idx: expected an int32 tensor [B,H,nT,topk]")
    topk = idx.shape[-1]
    _expect(idx, "idx", (B, Hkv if pooled else Hq, n_tiles(N), topk), torch.int32)
    extra = [("idx", idx)]
    if out is not None:
        _expect(out, "out", q.shape, q.dtype)
        extra.append(("out", out))
    _same_cuda_device([("q", q), ("k", k), ("v", v)] + extra)
    desc = prefill_desc(q, k, group_map, scale, pooled)
    out = torch.empty_like(q) if out is None else out
    ws, buf = _ws(ws, q.device, workspace_size(desc, topk, PREFILL), stream)
    _check(_lib.kascade_reuse_prefill(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), int(topk),
                                      _ptr(idx), _ptr(out), _ptr(buf), buf.numel(),
                                      _stream(stream)), "kascade_reuse_prefill")
    return out


# ------------------------------------------------------------------- stack --

def run_stack(mode, qs, ks, vs, topk, anchors, group_map=None, scale=None, outs=None,
              idx_buf=None, ws=None, stream=None, layer_events=None, pooled=False):
    """Run a layer stack; returns (outs, idx_buf). mode: DECODE or PREFILL.

    layer_events: optional list of torch.cuda.Event (timing enabled), one per
    layer, recorded on the stream after that layer's launches. pooled: one
    index set per KV head."""
    if mode not in (DECODE, PREFILL):
        raise ValueError("mode must be DECODE or PREFILL")
    L = len(qs)
    (B, Hq, Hkv, N, _), dev = _layers(qs, ks, vs, prefill=(mode == PREFILL))
    H = Hkv if pooled else Hq
    if mode == DECODE:
        desc = decode_desc(qs[0], ks[0], group_map, scale, pooled)
        shape = (B, H, topk)
    else:
        desc = prefill_desc(qs[0], ks[0], group_map, scale, pooled)
        shape = (B, H, n_tiles(N), topk)
    if outs is not None:
        if len(outs) != L:
            raise ValueError("outs: one tensor per layer (got %d for %d layers)" % (len(outs), L))
        _all_like(outs, "outs", qs[0].shape, qs[0].dtype, dev)
    if idx_buf is not None:
        _expect(idx_buf, "idx_buf", shape, torch.int32)
        _same_cuda_device([("qs[0]", qs[0]), ("idx_buf", idx_buf)])
    if layer_events is not None and len(layer_events) != L:
        raise ValueError("layer_events: one event per layer")
    outs = [torch.empty_like(q) for q in qs] if outs is None else outs
    if idx_buf is None:
        idx_buf = torch.empty(shape, dtype=torch.int32, device=dev)
    ws, buf = _ws(ws, dev, workspace_size(desc, topk, mode), stream)
    arr = lambda ts: (ctypes.c_void_p * L)(*[t.data_ptr() for t in ts])
    an = (ctypes.c_int32 * max(1, len(anchors)))(*[int(a) for a in anchors])
    if layer_events is None:
        _check(_lib.kascade_run_stack(ctypes.byref(desc), int(mode), L, arr(qs), arr(ks), arr(vs),
                                      int(topk), an, len(anchors), arr(outs), _ptr(idx_buf),
                                      _ptr(buf), buf.numel(), _stream(stream)), "kascade_run_stack")
    else:
        ev = (ctypes.c_void_p * L)(*[e.cuda_event for e in layer_events])
        _check(_lib.kascade_run_stack_profiled(ctypes.byref(desc), int(mode), L, arr(qs), arr(ks),
                                               arr(vs), int(topk), an, len(anchors), arr(outs),
                                               _ptr(idx_buf), _ptr(buf), buf.numel(),
                                               _stream(stream), ev), "kascade_run_stack_profiled")
    return outs, idx_buf


def kascade_attention(qs, ks, vs, topk, anchors, group_map=None, scale=None, pooled=False,
                      ws=None, stream=None):
    """One call over a layer stack, in the form the Kascade pages describe
    (euno.news summary, Practical Implications): per-layer lists qs, ks, vs,
    the Top-k size and the anchor layers. 3-D queries [B,Hq,d] are decode,
    4-D [B,Hq,N,d] causal prefill. Anchor layers compute exact attention and
    refresh the index sets, the layers after them reuse those sets, and
    layers before the first anchor run dense. Returns the per-layer outputs."""
    if len(qs) == 0:
        raise ValueError("qs: at least one layer")
    mode = DECODE if qs[0].dim() == 3 else PREFILL
    outs, _ = run_stack(mode, qs, ks, vs, topk, list(anchors), group_map=group_map, scale=scale,
                        ws=ws, stream=stream, pooled=pooled)
    return outs


# -------------------------------------------------------------- scheduling --

def layer_overlap(sets, n_bits, ws=None, stream=None):
    """sets: int32 [L, units, topk] on the device -> int64 counts [L, L]."""
    if not isinstance(sets, torch.Tensor) or sets.dim() != 3:
        raise ValueError("sets: expected an int32 tensor [L, units, topk]")
    L, units, k = sets.shape
    _expect(sets, "sets", (L, units, k), torch.int32)
    _same_cuda_device([("sets", sets)])
    counts = torch.empty(L, L, dtype=torch.int64, device=sets.device)
    nbytes = _lib.kascade_overlap_workspace_size(L, units, int(n_bits))
    ws, buf = _ws(ws, sets.device, nbytes, stream)
    _check(_lib.kascade_layer_overlap(_ptr(sets), L, units, k, int(n_bits), _ptr(counts),
                                      _ptr(buf), buf.numel(), _stream(stream)), "kascade_layer_overlap")
    return counts


def schedule_anchors(sim, n_anchors: int):
    """Host DP over a similarity matrix (sequence of rows); returns (anchors, objective)."""
    L = len(sim)
    flat = (ctypes.c_double * (L * L))(*[float(x) for row in sim for x in row])
    out = (ctypes.c_int32 * n_anchors)()
    obj = ctypes.c_double()
    _check(_lib.kascade_schedule_anchors(flat, L, int(n_anchors), out, ctypes.byref(obj)),
           "kascade_schedule_anchors")
    return list(out), obj.value


def calibrate(qs, ks, vs, topk, group_map=None, scale=None, ws=None, stream=None, pooled=False,
              similarity="overlap"):
    """Every layer as an anchor; returns (sim [L][L] list of lists, sets [L, B*H, topk]),
    H = Hq, or Hkv when pooled. similarity: "overlap" (Top-k set overlap) or
    "recall" (attention mass of layer l kept by layer i's set; 0 for i > l)."""
    if similarity not in ("overlap", "recall"):
        raise ValueError("similarity must be 'overlap' or 'recall'")
    recall = similarity == "recall"
    L = len(qs)
    (B, Hq, Hkv, _, _), dev = _layers(qs, ks, vs, prefill=False)
    desc = decode_desc(qs[0], ks[0], group_map, scale, pooled)
    H = Hkv if pooled else Hq
    outs = [torch.empty_like(q) for q in qs]
    sets = torch.empty(L, B * H, topk, dtype=torch.int32, device=dev)
    size_fn = (_lib.kascade_calibrate_recall_workspace_size if recall
               else _lib.kascade_calibrate_workspace_size)
    nbytes = size_fn(ctypes.byref(desc), int(topk), L)
    if nbytes == 0:
        raise KascadeError(INVALID_ARG, "calibration workspace size")
    ws, buf = _ws(ws, dev, nbytes, stream)
    arr = lambda ts: (ctypes.c_void_p * L)(*[t.data_ptr() for t in ts])
    sim = (ctypes.c_double * (L * L))()
    fn = _lib.kascade_calibrate_recall if recall else _lib.kascade_calibrate
    _check(fn(ctypes.byref(desc), L, arr(qs), arr(ks), arr(vs), int(topk), arr(outs), _ptr(sets),
              sim, _ptr(buf), buf.numel(), _stream(stream)),
           "kascade_calibrate_recall" if recall else "kascade_calibrate")
    return [[sim[i * L + j] for j in range(L)] for i in range(L)], sets
