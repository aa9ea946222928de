"""Seeded synthetic attention workloads.

This module only draws inputs. It holds none of the attention, Top-k or
scheduling arithmetic, so the CPU oracle and the CUDA path can both consume
what it produces without sharing any of the method's code.

Recipe (Kascade, "A Practical Sparse Attention Method for Long-Context LLM
Inference": the Abstract says post-softmax attention is sparse and the
identity of high-weight keys is stable across nearby layers; the generator
plants both properties):

* layer 0: q, k, v ~ N(0, 1) in fp32 from a ``torch.Generator`` seeded with
  ``seed``;
* planting: for every (sequence b, query head h), ``n_plants`` distinct key
  positions drawn from [1, N) get ``plant_strength * q_h / |q_h|`` added to
  the key row of KV head g(h) (position 0 is kept for the sink). Heads of one
  group add up where they collide. For prefill the direction is the query of
  the last position;
* sink (when enabled): key row 0 of KV head g gets ``4 * u_g`` added, where
  u_g is the normalised sum of the group's (last-position) query vectors;
* layer l > 0: X_l = rho_l * X_{l-1} + sqrt(1 - rho_l^2) * Z for X in
  {q, k, v}, Z fresh N(0, 1), applied to the planted previous layer; plants
  and sink are not re-applied, so they decay geometrically;
* every layer is rounded to the storage dtype (bf16 round-to-nearest-even, or
  kept fp32) after all additions; the chain keeps the unrounded fp32 state.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Iterator, Optional, Sequence, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    mode: str                 # "decode" or "prefill"
    n_layers: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    kv_len: int               # N: KV-cache length (decode) or sequence length (prefill)
    topk: int                 # k
    anchors: Tuple[int, ...]
    dtype: str                # "f32" or "bf16"
    n_plants: int
    plant_strength: float = 3.0
    sink: bool = True
    rho: float = 0.9
    rho_range: Optional[Tuple[float, float]] = None   # per-layer rho ~ U[a, b] when set
    seed: int = 1000
    # seed of the per-layer rho draw when it differs from `seed`: evaluation
    # sequences of a schedule are fresh draws on the calibration's rhos
    rho_seed: Optional[int] = None
    tile: int = 128

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def group_map(n_q_heads: int, n_kv_heads: int):
    """Default GQA map: query head h reads KV head h // (Hq / Hkv)."""
    g = n_q_heads // n_kv_heads
    return [h // g for h in range(n_q_heads)]


def layer_rhos(w: Workload) -> list:
    """Per-layer chain coefficients; rho_0 is unused."""
    if w.rho_range is None:
        return [w.rho] * w.n_layers
    gen = torch.Generator(device="cpu").manual_seed(
        (w.seed if w.rho_seed is None else w.rho_seed) + 7919)
    a, b = w.rho_range
    u = torch.rand(w.n_layers, generator=gen, dtype=torch.float64)
    return [float(a + (b - a) * x) for x in u]


def _shapes(w: Workload):
    B, Hq, Hkv, d, N = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.kv_len
    if w.mode == "decode":
        return (B, Hq, d), (B, Hkv, N, d)
    return (B, Hq, N, d), (B, Hkv, N, d)


def _plant(w: Workload, q, k, gen, gmap):
    B, Hq, N = w.batch, w.n_q_heads, w.kv_len
    qlast = q if w.mode == "decode" else q[:, :, -1, :]          # [B, Hq, d]
    qdir = qlast / qlast.norm(dim=-1, keepdim=True)
    if w.n_plants > 0:
        P = min(w.n_plants, N - 1)
        # P distinct positions in [1, N) per (b, h): the P largest of N-1 uniforms
        r = torch.rand(B, Hq, N - 1, generator=gen, device=q.device)
        pos = r.topk(P, dim=-1).indices + 1                     # [B, Hq, P]
        for b in range(B):
            for h in range(Hq):
                row = (w.plant_strength * qdir[b, h]).expand(P, -1)
                k[b, gmap[h]].index_add_(0, pos[b, h], row)
    if w.sink:
        for b in range(B):
            for g in range(w.n_kv_heads):
                hs = [h for h in range(Hq) if gmap[h] == g]
                u = qlast[b, hs].sum(dim=0)
                k[b, g, 0] += 4.0 * u / u.norm()


def layers(w: Workload, device="cpu", seed: Optional[int] = None,
           gmap: Optional[Sequence[int]] = None) -> Iterator[Tuple[torch.Tensor, torch.Tensor, torch.Tensor]]:
    """Yield (q, k, v) for layer 0, 1, ... in the storage dtype, on ``device``."""
    seed = w.seed if seed is None else seed
    gmap = list(gmap) if gmap is not None else group_map(w.n_q_heads, w.n_kv_heads)
    gen = torch.Generator(device=device).manual_seed(seed)
    qs, ks = _shapes(w)
    rhos = layer_rhos(w)
    q = torch.randn(qs, generator=gen, device=device, dtype=torch.float32)
    k = torch.randn(ks, generator=gen, device=device, dtype=torch.float32)
    v = torch.randn(ks, generator=gen, device=device, dtype=torch.float32)
    _plant(w, q, k, gen, gmap)
    for layer in range(w.n_layers):
        if layer > 0:
            rho = rhos[layer]
            c = math.sqrt(1.0 - rho * rho)
            for x in (q, k, v):
                z = torch.randn(x.shape, generator=gen, device=device, dtype=torch.float32)
                x.mul_(rho).add_(z, alpha=c)
                del z
        # copy=True: the fp32 state is updated in place for the next layer
        yield (q.to(w.torch_dtype, copy=True), k.to(w.torch_dtype, copy=True),
               v.to(w.torch_dtype, copy=True))


def make_layers(w: Workload, device="cpu", seed: Optional[int] = None, gmap=None):
    """All layers at once: lists q[L], k[L], v[L]."""
    qs, ks, vs = [], [], []
    for q, k, v in layers(w, device=device, seed=seed, gmap=gmap):
        qs.append(q)
        ks.append(k)
        vs.append(v)
    return qs, ks, vs


def n_tiles(n: int, tile: int = 128) -> int:
    return (n + tile - 1) // tile
