"""Run one attention layer kind a few times on synthetic inputs (for profilers).

    python -m long_context_anchor_gb300.runcase KIND [--batch B] [--kv-len N]
        [--heads HQ HKV] [--head-dim D] [--topk K] [--reps R] [--pooled]

KIND: dense_decode, anchor_decode, anchor_decode_fused, reuse_decode, topk,
dense_prefill, anchor_prefill, reuse_prefill. Defaults are the Llama-3.1-8B attention shape
with batch 2 (decode: about 0.5 GB of K/V per layer, larger than L2), so a
profiler capture of one launch stays small. Inputs are drawn once; every
repetition runs the same launch sequence. --pooled uses one index set per KV
head (anchor and reuse kinds).
"""
import argparse

import torch

from . import kascade as K


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("kind")
    ap.add_argument("--batch", type=int, default=2)
    ap.add_argument("--kv-len", type=int, default=32768)
    ap.add_argument("--heads", type=int, nargs=2, default=(32, 8))
    ap.add_argument("--head-dim", type=int, default=128)
    ap.add_argument("--topk", type=int, default=0, help="default kv_len // 8")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--pooled", action="store_true", help="one index set per KV head")
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(7)
    B, N, (Hq, Hkv), d = a.batch, a.kv_len, a.heads, a.head_dim
    k_top = a.topk or max(1, N // 8)
    bf = torch.bfloat16
    if "decode" in a.kind or a.kind == "topk":
        q = torch.randn(B, Hq, d, generator=g, device=dev).to(bf)
    else:
        q = torch.randn(B, Hq, N, d, generator=g, device=dev).to(bf)
    k = torch.randn(B, Hkv, N, d, generator=g, device=dev).to(bf)
    v = torch.randn(B, Hkv, N, d, generator=g, device=dev).to(bf)
    ws = K.Workspace(dev)
    idx = None
    pl = a.pooled
    if a.kind == "reuse_decode":
        _, idx = K.anchor_decode(q, k, v, k_top, ws=ws, pooled=pl)
    if a.kind == "reuse_prefill":
        _, idx = K.anchor_prefill(q, k, v, k_top, ws=ws, pooled=pl)
    scores = None
    if a.kind == "topk":
        scores = torch.randn(B * Hq, N, generator=g, device=dev)
    torch.cuda.synchronize()
    for _ in range(a.reps):
        if a.kind == "dense_decode":
            K.dense_decode(q, k, v, ws=ws)
        elif a.kind == "anchor_decode":
            K.anchor_decode(q, k, v, k_top, ws=ws, pooled=pl)
        elif a.kind == "anchor_decode_fused":
            K.anchor_decode(q, k, v, k_top, ws=ws, fused=True)
        elif a.kind == "reuse_decode":
            K.reuse_decode(q, k, v, idx, ws=ws, pooled=pl)
        elif a.kind == "topk":
            K.topk(scores, k_top, ws=ws)
        elif a.kind == "dense_prefill":
            K.dense_prefill(q, k, v, ws=ws)
        elif a.kind == "anchor_prefill":
            K.anchor_prefill(q, k, v, k_top, ws=ws, pooled=pl)
        elif a.kind == "reuse_prefill":
            K.reuse_prefill(q, k, v, idx, ws=ws, pooled=pl)
        else:
            raise SystemExit("unknown kind " + a.kind)
    torch.cuda.synchronize()
    err = ws.device_error()
    if err != K.OK:
        raise SystemExit("device error: " + K.status_string(err))
    print("ok", a.kind)


if __name__ == "__main__":
    main()
