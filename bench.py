#!/usr/bin/env python
"""Benchmark: Kascade decode attention on the Llama-3.1-8B attention shape.

Workload (one step = one pass of the whole decode stack): 32 layers, batch 8,
32 query / 8 KV heads, head_dim 128, bf16, KV cache N = 32768 per sequence,
one query per sequence, Top-k k = 4096, anchors {0, 4, ..., 28}; seeded
synthetic inputs (planted heavy keys, attention sink, cross-layer
correlation 0.9). Each layer's K/V (1.07 GB) is distinct and far larger than
L2, so no flush is needed between layers or steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). `value` is decode attention time per layer in
microseconds (lower is better) for the Kascade stack; the same line carries
the library's own dense-attention stack on the same inputs, HBM GB/s, the
roofline of the dominant kernel, an end-to-end number through the public API
with host buffers, and the CPU oracle timed on the host cores.
The line also carries the prefill stack (Llama-3.1-8B shape, N=16384) and the
long-context decode stack (gpt-oss-20b-like shape: 24 layers, 64/8 heads,
d=64, B=4, N=131072, k=8192), each against the library's own dense kernels
with its own roofline, end-to-end pass and oracle sample, and the schedule
sweep: six anchors chosen by the DP from calibration on four sequences, then
decode at batch 16 and prefill at N = 4096, 16384 and 65536 with those
anchors. ``--impl reference`` times the CPU oracle itself on a bounded sample.
"""
import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn µs/layer + HBM GB/s at 32K ctx; prefill attn TFLOP/s; vs own dense"

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch from one
# ncu capture of the kernel as it stands (profiles/<kernel>_*.md); None when no
# capture of the current kernel at the bench's size exists.
TRAFFIC = {
    "k_decode_union_bf16": 450.881e6,   # profiles/k_decode_union_bf16_llama8b_b8_n32768.md
    "k_prefill_fa2_reuse": 383.524e6,   # profiles/k_prefill_fa2_reuse_n16384.md
    # captured at B=1 (8 of the 32 units) and scaled by units to B=4:
    # profiles/k_decode_union_bf16_gptoss_b4_n131072.md
    "k_decode_union_bf16_long": 4 * 111.014e6,
}
UNIT = "us/layer"
NOMINAL_HBM_GBS = 8000.0   # the ~8 TB/s HBM3e figure the decode targets are quoted against


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons.

    The sampler runs from `start()` to `stop()`; `begin()`/`end()` bracket each
    timed region, and `stop()` keeps only the samples taken inside a region
    (widened by one sampling period, so that regions shorter than the period
    still get their nearest sample)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 100

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.path = None
        self.windows = []

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)   # let the first samples arrive before the first region

    def begin(self):
        self.windows.append([datetime.datetime.now(), None])

    def end(self):
        self.windows[-1][1] = datetime.datetime.now()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(2 * self.PERIOD_MS / 1e3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        pad = datetime.timedelta(milliseconds=self.PERIOD_MS)
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                sample = (float(parts[1]), float(parts[2]), parts[5:9])
            except ValueError:
                continue
            if any(b - pad <= ts <= e + pad for b, e in self.windows if e is not None):
                rows.append(sample)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i] == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "samples": len(rows),
                "timed_regions": len(self.windows), "reasons": reasons}


# ---------------------------------------------------------- CPU oracle leg --

def _oracle_group(task):
    """One (sequence, KV head) group of one layer through the float64 oracle.

    task = (kind, q [G,d], K [N,d], V [N,d], idx [G,k] or None, k, scale).
    Runs in a spawned worker with single-threaded BLAS.
    """
    import numpy as np
    from oracle import attention as A
    kind, q, Kg, Vg, idx, k, scale = task
    t0 = time.perf_counter()
    G = q.shape[0]
    qd = q[None].astype(np.float64)                    # [1, G, d]
    Kd = Kg[None, None].astype(np.float64)             # [1, 1, N, d]
    Vd = Vg[None, None].astype(np.float64)
    gm = [0] * G
    if kind == "anchor":
        A.anchor_decode(qd, Kd, Vd, k, gm, scale)
    else:
        A.sparse_decode(qd, Kd, Vd, idx[None], gm, scale)
    return time.perf_counter() - t0


def oracle_sample_tasks(w, layers_dev, n_groups, seed=0):
    """Host copies of n_groups (sequence, KV head) groups of layer 0 (anchor) and
    layer 1 (reuse, using the oracle's own layer-0 sets computed in the worker
    order). Returns (anchor_tasks, reuse_tasks)."""
    import numpy as np
    import torch
    from oracle.topk import topk_indices
    (q0, k0, v0), (q1, k1, v1) = layers_dev
    rng = np.random.default_rng(seed)
    G = w.n_q_heads // w.n_kv_heads
    scale = 1.0 / np.sqrt(w.head_dim)
    units = [(int(rng.integers(w.batch)), int(rng.integers(w.n_kv_heads))) for _ in range(n_groups)]
    f32 = lambda t: t.float().cpu().numpy()
    at, rt = [], []
    for b, g in units:
        hs = list(range(g * G, (g + 1) * G))
        qa, Ka, Va = f32(q0[b, hs]), f32(k0[b, g]), f32(v0[b, g])
        at.append(("anchor", qa, Ka, Va, None, w.topk, scale))
        # sets for the reuse task: oracle Top-k of this group's layer-0 logits
        s = scale * (Ka.astype(np.float64) @ qa.astype(np.float64).T)   # [N, G]
        idx = np.stack([topk_indices(s[:, i], w.topk) for i in range(G)])
        rt.append(("reuse", f32(q1[b, hs]), f32(k1[b, g]), f32(v1[b, g]), idx, w.topk, scale))
    return at, rt


def time_oracle(w, layers_dev, n_groups, reps=1):
    """Wall time of the oracle on the sample, extrapolated to microseconds per
    layer of the stack (anchor/reuse mix of the schedule). Returns a dict."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    at, rt = oracle_sample_tasks(w, layers_dev, n_groups)
    cores = os.cpu_count() or 1
    old = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in old:
        os.environ[k] = "1"
    try:
        with ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")) as ex:
            list(ex.map(_oracle_group, at[:1]))           # start the workers
            ta, tr = [], []
            for _ in range(reps):
                t0 = time.perf_counter()
                list(ex.map(_oracle_group, at))
                ta.append(time.perf_counter() - t0)
                t0 = time.perf_counter()
                list(ex.map(_oracle_group, rt))
                tr.append(time.perf_counter() - t0)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    groups_per_layer = w.batch * w.n_kv_heads
    n_anchor = len(w.anchors)
    n_reuse = w.n_layers - n_anchor
    per_a = statistics.median(ta) * groups_per_layer / n_groups
    per_r = statistics.median(tr) * groups_per_layer / n_groups
    us = 1e6 * (n_anchor * per_a + n_reuse * per_r) / w.n_layers
    return {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle", "extrapolated": True,
            "sample": "%d of %d (sequence, KV head) groups of one anchor layer and one reuse "
                      "layer (float64 numpy, one process per core, single-threaded BLAS); "
                      "extrapolated to the %d-anchor / %d-reuse stack" %
                      (n_groups, groups_per_layer, n_anchor, n_reuse),
            "anchor_layer_s": per_a, "reuse_layer_s": per_r}


def _oracle_prefill_unit(task):
    """One (head, 128-row tile) unit of one prefill layer through the float64
    oracle, in a spawned worker with single-threaded BLAS.

    task = (kind, Q [L_t, d], K [L_t, d], V [L_t, d], t, k or set, scale): the
    causal prefix up to the tile's last row. Returns (seconds, set or None)."""
    import numpy as np
    from oracle import attention as A
    kind, Q, Kt, Vt, t, arg, scale = task
    t0 = time.perf_counter()
    q4, k4, v4 = (x[None, None].astype(np.float64) for x in (Q, Kt, Vt))
    if kind == "anchor":
        _, idx, _ = A.anchor_prefill_tile(q4, k4, v4, 0, 0, t, arg, [0], scale)
    else:
        A.sparse_prefill_tile(q4, k4, v4, arg, 0, 0, t, [0], scale)
        idx = None
    return time.perf_counter() - t0, idx


def time_oracle_prefill(w, layers_dev, n_units, reps=1, seed=0):
    """Wall time of the oracle on a seed-fixed sample of (head, tile) units of
    one anchor prefill layer (exact rows, tile weights, Top-k) and one reuse
    layer (over the oracle's own sets), always including the first and the
    last tile, one process per host core; extrapolated by unit count to
    milliseconds per stack of the schedule."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    (q0, k0, v0), (q1, k1, v1) = layers_dev
    N, T = w.kv_len, w.tile
    nT = (N + T - 1) // T
    G = w.n_q_heads // w.n_kv_heads
    scale = 1.0 / np.sqrt(w.head_dim)
    rng = np.random.default_rng(seed)
    units = [(0, 0), (w.n_q_heads - 1, nT - 1)] + \
        [(int(rng.integers(w.n_q_heads)), int(rng.integers(nT))) for _ in range(n_units - 2)]
    f32 = lambda x: x.float().cpu().numpy()
    at, rq = [], []
    for h, t in units:
        L = min(N, T * (t + 1))
        g = h // G
        at.append(("anchor", f32(q0[0, h, :L]), f32(k0[0, g, :L]), f32(v0[0, g, :L]), t, w.topk,
                   scale))
        rq.append((f32(q1[0, h, :L]), f32(k1[0, g, :L]), f32(v1[0, g, :L]), t))
    cores = os.cpu_count() or 1
    old = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in old:
        os.environ[k] = "1"
    try:
        with ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")) as ex:
            list(ex.map(_oracle_prefill_unit, at[:1]))        # start the workers
            ta, tr = [], []
            for _ in range(reps):
                t0 = time.perf_counter()
                sets = [r[1] for r in ex.map(_oracle_prefill_unit, at)]
                ta.append(time.perf_counter() - t0)
                rt = [("reuse", Q, Kt, Vt, t, sel, scale) for (Q, Kt, Vt, t), sel in zip(rq, sets)]
                t0 = time.perf_counter()
                list(ex.map(_oracle_prefill_unit, rt))
                tr.append(time.perf_counter() - t0)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    units_per_layer = w.batch * w.n_q_heads * nT
    n_anchor = len(w.anchors)
    n_reuse = w.n_layers - n_anchor
    per_a = statistics.median(ta) * units_per_layer / n_units
    per_r = statistics.median(tr) * units_per_layer / n_units
    return {"value": 1e3 * (n_anchor * per_a + n_reuse * per_r), "unit": "ms/stack",
            "cores": cores, "kind": "oracle", "extrapolated": True,
            "sample": "%d of %d (query head, 128-row tile) units, first and last tile included, "
                      "of one anchor layer and one reuse layer (float64 numpy, one process per "
                      "core, single-threaded BLAS); extrapolated by unit count to the "
                      "%d-anchor / %d-reuse stack" % (n_units, units_per_layer, n_anchor, n_reuse),
            "anchor_layer_s": per_a, "reuse_layer_s": per_r}


# --------------------------------------------------------------- GPU legs --

def decode_bytes(w, union_rows_per_anchor):
    """Algorithmic HBM bytes per layer kind (bf16 K/V rows of 2*d bytes each).

    dense  : every K and V row once + q read + out write;
    anchor : dense + fp32 logits spill written and read back by the Top-k
             + int32 index sets written (+ read once to build the union plan);
    reuse  : K and V rows of the union of the group's sets, once each, + one
             4-byte plan entry per union row + q + out.
    """
    d, B, Hq, Hkv, N, k = w.head_dim, w.batch, w.n_q_heads, w.n_kv_heads, w.kv_len, w.topk
    qo = 2 * B * Hq * d * 2
    dense = B * Hkv * N * 2 * d * 2 + qo
    reuse = [u * (2 * d * 2 + 4) + qo for u in union_rows_per_anchor]
    anchor = [dense + 2 * B * Hq * N * 4 + 2 * B * Hq * k * 4 + 4 * u for u in union_rows_per_anchor]
    return dense, anchor, reuse


def pooled_decode_bytes(w):
    """Algorithmic HBM bytes per layer with one index set per (sequence, KV head).

    anchor: dense + fp32 logits spill written and read back + the pooled
            weights written and read by the Top-k + index sets written;
    reuse : K and V rows of the group's set (k rows, no union needed) + the
            4-byte set entry of each row (the set is the gather list) + q + out.
    """
    d, B, Hq, Hkv, N, k = w.head_dim, w.batch, w.n_q_heads, w.n_kv_heads, w.kv_len, w.topk
    qo = 2 * B * Hq * d * 2
    dense = B * Hkv * N * 2 * d * 2 + qo
    anchor = dense + 2 * B * Hq * N * 4 + 2 * B * Hkv * N * 4 + B * Hkv * k * 4
    reuse = B * Hkv * k * (2 * d * 2 + 4) + qo
    return anchor, reuse


def union_rows(idx, w):
    """Rows of the per-(sequence, KV head) union of the group's index sets."""
    import torch
    B, Hq, k = idx.shape
    G = w.n_q_heads // w.n_kv_heads
    mark = torch.zeros(B, w.n_kv_heads, w.kv_len, dtype=torch.bool, device=idx.device)
    for h in range(Hq):
        mark[:, h // G].scatter_(1, idx[:, h].long(), True)
    return int(mark.sum().item())


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def max_over_ranks(values, world, device=None):
    """Element-wise maximum of a list of floats over all ranks (one all_reduce);
    the list itself when there is one rank."""
    values = [float(v) for v in values]
    if world <= 1:
        return values
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def prefill_flops(w, topk_sizes=None):
    """Algorithmic FLOPs per layer kind for causal prefill (bf16 MMAs).

    dense : QK^T and PV over the causal pairs, 4 * d * Hq * N(N+1)/2;
    anchor: dense + one more QK^T pass for the tile weights (1.5 x dense);
    reuse : QK^T and PV of every 128-row tile against its k_t saved keys,
            4 * d * Hq * sum_t rows_t * k_t.
    """
    N, d, Hq, k, T = w.kv_len, w.head_dim, w.n_q_heads, w.topk, w.tile
    pairs = N * (N + 1) // 2
    dense = 4 * d * Hq * pairs * w.batch
    anchor = dense * 3 // 2
    nT = (N + T - 1) // T
    tile_pairs = sum(min(N, T * (t + 1)) - T * t for t in range(nT))
    reuse = 4 * d * Hq * w.batch * sum((min(N, T * (t + 1)) - T * t) * min(k, min(N, T * (t + 1)))
                                       for t in range(nT))
    del tile_pairs
    return dense, anchor, reuse


# ---------------------------------------------------------- end to end legs --

def decode_e2e(K, w, q_all, k_all, v_all, out_all, anchors, idx_buf, ws, stream, steps, warmup,
               world, dev):
    """Decode stack end to end through kascade_run_stack with host buffers.

    Each step copies every layer's new query and the newest K/V row
    (position N-1) from pinned host memory, runs the stack and reads all
    outputs back. The copies run on a second stream into two sets of device
    staging buffers, so step s+1's inputs travel while step s computes and
    step s's outputs travel while step s+1 computes; every step's own copies
    stay inside the timed region (the first upload and the last download are
    not hidden)."""
    import torch
    L, N = w.n_layers, w.kv_len
    q_host = q_all.cpu().pin_memory()
    knew_host = k_all[:, :, :, N - 1].contiguous().cpu().pin_memory()
    vnew_host = v_all[:, :, :, N - 1].contiguous().cpu().pin_memory()
    out_host = [torch.empty(out_all.shape, dtype=out_all.dtype).pin_memory() for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)
    down_stream = copy_stream   # the copies are small: one stream for both directions
    q_stage = [torch.empty_like(q_all) for _ in range(2)]
    kn_stage = [torch.empty(knew_host.shape, dtype=knew_host.dtype, device=dev) for _ in range(2)]
    vn_stage = [torch.empty(vnew_host.shape, dtype=vnew_host.dtype, device=dev) for _ in range(2)]
    out_stage = [torch.empty_like(out_all) for _ in range(2)]
    ks, vs = list(k_all), list(v_all)
    up_done = [torch.cuda.Event() for _ in range(2)]
    step_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]
    slot_used = [False, False]

    def upload(slot):
        with torch.cuda.stream(copy_stream):
            if slot_used[slot]:
                copy_stream.wait_event(down_done[slot])   # the slot's previous step is done
            q_stage[slot].copy_(q_host, non_blocking=True)
            kn_stage[slot].copy_(knew_host, non_blocking=True)
            vn_stage[slot].copy_(vnew_host, non_blocking=True)
            up_done[slot].record(copy_stream)
        slot_used[slot] = True

    def compute(slot):
        stream.wait_event(up_done[slot])
        k_all[:, :, :, N - 1].copy_(kn_stage[slot])
        v_all[:, :, :, N - 1].copy_(vn_stage[slot])
        K.run_stack(K.DECODE, list(q_stage[slot]), ks, vs, w.topk, anchors,
                    outs=list(out_stage[slot]), idx_buf=idx_buf, ws=ws)
        step_done[slot].record(stream)

    def download(slot):
        with torch.cuda.stream(down_stream):
            down_stream.wait_event(step_done[slot])
            out_host[slot].copy_(out_stage[slot], non_blocking=True)
            down_done[slot].record(down_stream)

    def run(n):
        upload(0)
        for st in range(n):
            if st + 1 < n:
                upload((st + 1) % 2)
            compute(st % 2)
            download(st % 2)
        stream.wait_event(down_done[(n - 1) % 2])

    run(warmup)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    down_stream.wait_event(e0)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize()
    # the outputs that came back are the stack's outputs for these inputs
    assert torch.equal(out_host[(steps - 1) % 2], out_stage[(steps - 1) % 2].cpu())
    assert ws.device_error() == K.OK
    ms = max_over_ranks([e0.elapsed_time(e1) / steps], world, dev)[0]
    return {"value": round(1e3 * ms / L, 3), "unit": UNIT,
            "h2d_bytes_per_step": int(q_host.numel() * 2 + 2 * knew_host.numel() * 2),
            "d2h_bytes_per_step": int(out_host[0].numel() * 2),
            "copies": "second stream, double-buffered staging; D2D scatter of the new K/V rows "
                      "per step"}


def prefill_e2e(K, w, qs, ks, vs, anchors, ws, stream, steps, warmup, world, dev,
                copy_streams=2):
    """Prefill stack end to end through kascade_run_stack with host buffers.

    Each step copies every layer's Q, K and V (the whole prompt) from pinned
    host memory, runs the stack and reads every layer's output back; a second
    stream and two sets of device staging buffers overlap step s+1's upload
    and step s-1's download with step s's compute, and every step's own
    copies stay inside the timed region."""
    import torch
    L = w.n_layers
    stack_h = lambda ts: torch.stack(ts).cpu().pin_memory()
    q_host, k_host, v_host = stack_h(qs), stack_h(ks), stack_h(vs)
    out_host = [torch.empty(q_host.shape, dtype=q_host.dtype).pin_memory() for _ in range(2)]
    # uploads on one copy stream; downloads on their own (copy_streams=2), so
    # that both directions of the host link carry data at once (48 against
    # 54 ms per stack with one stream for both, measured on one box), or on
    # the same one (copy_streams=1)
    copy_stream = torch.cuda.Stream(device=dev)
    down_stream = torch.cuda.Stream(device=dev) if copy_streams == 2 else copy_stream
    stage = [[torch.empty(h.shape, dtype=h.dtype, device=dev) for h in (q_host, k_host, v_host)]
             for _ in range(2)]
    out_stage = [torch.empty(q_host.shape, dtype=q_host.dtype, device=dev) for _ in range(2)]
    up_done = [torch.cuda.Event() for _ in range(2)]
    step_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]
    slot_used = [False, False]
    nT = (w.kv_len + w.tile - 1) // w.tile
    idx_buf = torch.empty(w.batch, w.n_q_heads, nT, w.topk, dtype=torch.int32, device=dev)

    def upload(slot):
        with torch.cuda.stream(copy_stream):
            if slot_used[slot]:
                copy_stream.wait_event(down_done[slot])
            for dst, src in zip(stage[slot], (q_host, k_host, v_host)):
                dst.copy_(src, non_blocking=True)
            up_done[slot].record(copy_stream)
        slot_used[slot] = True

    def compute(slot):
        stream.wait_event(up_done[slot])
        qd, kd, vd = stage[slot]
        K.run_stack(K.PREFILL, list(qd), list(kd), list(vd), w.topk, anchors,
                    outs=list(out_stage[slot]), idx_buf=idx_buf, ws=ws)
        step_done[slot].record(stream)

    def download(slot):
        with torch.cuda.stream(down_stream):
            down_stream.wait_event(step_done[slot])
            out_host[slot].copy_(out_stage[slot], non_blocking=True)
            down_done[slot].record(down_stream)

    def run(n):
        upload(0)
        for st in range(n):
            if st + 1 < n:
                upload((st + 1) % 2)
            compute(st % 2)
            download(st % 2)
        stream.wait_event(down_done[(n - 1) % 2])

    run(warmup)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    down_stream.wait_event(e0)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize()
    assert torch.equal(out_host[(steps - 1) % 2], out_stage[(steps - 1) % 2].cpu())
    assert ws.device_error() == K.OK
    ms = max_over_ranks([e0.elapsed_time(e1) / steps], world, dev)[0]
    h2d = sum(h.numel() * h.element_size() for h in (q_host, k_host, v_host))
    res = {"value": round(ms, 3), "unit": "ms/stack", "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(out_host[0].numel() * out_host[0].element_size()),
           "copies": ("second stream" if copy_streams == 1 else "upload and download streams") +
                     ", double-buffered staging of every layer's Q, K, V and output"}
    del stage, out_stage, out_host, q_host, k_host, v_host
    torch.cuda.empty_cache()
    return res


def run_prefill(args, dev, world, stream, clocks):
    """Prefill stack of the Llama-3.1-8B shape at N = 16384 (32 layers,
    anchors every 4th layer): Kascade vs the library's own dense prefill."""
    import torch
    import torch.distributed as dist
    from long_context_anchor_gb300 import configs
    from long_context_anchor_gb300 import kascade as K
    from long_context_anchor_gb300.workloads import make_layers
    w = configs.LLAMA8B_PREFILL_16K
    L = w.n_layers
    qs, ks, vs = make_layers(w, device=dev)
    outs = [torch.empty_like(q) for q in qs]
    nT = (w.kv_len + 127) // 128
    idx_buf = torch.empty(w.batch, w.n_q_heads, nT, w.topk, dtype=torch.int32, device=dev)
    idx_pool = torch.empty(w.batch, w.n_kv_heads, nT, w.topk, dtype=torch.int32, device=dev)
    ws = K.Workspace(dev)
    anchors = list(w.anchors)

    def timed(anch, steps, pooled=False):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(L + 1)] for _ in range(steps)]
        for row in evs:
            for e in row:
                e.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        for s in range(steps):
            evs[s][0].record(stream)
            K.run_stack(K.PREFILL, qs, ks, vs, w.topk, anch, outs=outs,
                        idx_buf=idx_pool if pooled else idx_buf, ws=ws,
                        layer_events=evs[s][1:], pooled=pooled)
        torch.cuda.synchronize()
        per = [[evs[s][l].elapsed_time(evs[s][l + 1]) for l in range(L)] for s in range(steps)]
        total = sum(evs[s][0].elapsed_time(evs[s][L]) for s in range(steps))
        return total, per

    for _ in range(args.warmup):
        K.run_stack(K.PREFILL, qs, ks, vs, w.topk, anchors, outs=outs, idx_buf=idx_buf, ws=ws)
        K.run_stack(K.PREFILL, qs, ks, vs, w.topk, [], outs=outs, idx_buf=idx_buf, ws=ws)
    torch.cuda.synchronize()
    assert ws.device_error() == K.OK
    steps = max(1, args.steps // 2)
    clocks.begin()
    tot_k, per_k = timed(anchors, steps)
    tot_d, per_d = timed([], steps)
    clocks.end()
    tot_k, tot_d = max_over_ranks([tot_k, tot_d], world, dev)
    ms_k, ms_d = tot_k / steps, tot_d / steps
    reuse_layers = [l for l in range(L) if l not in anchors]
    anchor_ms = statistics.mean(per_k[s][l] for s in range(steps) for l in anchors)
    reuse_ms = statistics.mean(per_k[s][l] for s in range(steps) for l in reuse_layers)
    dense_ms = ms_d / L
    f_dense, f_anchor, f_reuse = prefill_flops(w)
    _, tf_burst, src = load_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tf_sust = float(json.load(f)["bf16_tflops_sustained"])
    except (OSError, KeyError, ValueError):
        tf_sust = 1700.0
    res = {
        "workload": w.name, "layers": L, "kv_len": w.kv_len, "topk": w.topk, "anchors": anchors,
        "kascade_ms_per_stack": round(ms_k, 3), "dense_ms_per_stack": round(ms_d, 3),
        "speedup_vs_own_dense": round(ms_d / ms_k, 3),
        "anchor_layer_us": round(1e3 * anchor_ms, 1), "reuse_layer_us": round(1e3 * reuse_ms, 1),
        "dense_layer_us": round(1e3 * dense_ms, 1),
        "dense_tflops": round(f_dense / (dense_ms * 1e-3) / 1e12, 1),
        "anchor_tflops": round(f_anchor / (anchor_ms * 1e-3) / 1e12, 1),
        "reuse_tflops": round(f_reuse / (reuse_ms * 1e-3) / 1e12, 1),
        "stack_tflops": round((len(anchors) * f_anchor + len(reuse_layers) * f_reuse) /
                              (ms_k * 1e-3) / 1e12, 1),
        "flops_per_layer": {"dense": f_dense, "anchor": f_anchor, "reuse": f_reuse},
        "peak_bf16_tflops_sustained": tf_sust, "peak_bf16_tflops_burst": tf_burst,
        "peak_source": src,
    }
    if not args.no_pooled:
        # GQA-pooled tile sets (one per KV head) on the same inputs
        K.run_stack(K.PREFILL, qs, ks, vs, w.topk, anchors, outs=outs, idx_buf=idx_pool, ws=ws,
                    pooled=True)
        torch.cuda.synchronize()
        assert ws.device_error() == K.OK
        clocks.begin()
        tot_p, per_p = timed(anchors, steps, pooled=True)
        clocks.end()
        tot_p = max_over_ranks([tot_p], world, dev)[0]
        ms_p = tot_p / steps
        pa = statistics.mean(per_p[s][l] for s in range(steps) for l in anchors)
        pr = statistics.mean(per_p[s][l] for s in range(steps) for l in reuse_layers)
        res["pooled"] = {"index_sets": "one per (KV head, tile): group sums of tile weights",
                         "kascade_ms_per_stack": round(ms_p, 3),
                         "speedup_vs_own_dense": round(ms_d / ms_p, 3),
                         "anchor_layer_us": round(1e3 * pa, 1), "reuse_layer_us": round(1e3 * pr, 1),
                         "reuse_tflops": round(f_reuse / (pr * 1e-3) / 1e12, 1),
                         "reuse_frac_of_sustained": round(f_reuse / (pr * 1e-3) / 1e12 / tf_sust, 4),
                         "gpu_launches": steps * (4 * len(anchors) + len(reuse_layers))}
    res["dense_frac_of_sustained"] = round(res["dense_tflops"] / tf_sust, 4)
    res["anchor_frac_of_sustained"] = round(res["anchor_tflops"] / tf_sust, 4)
    res["reuse_frac_of_sustained"] = round(res["reuse_tflops"] / tf_sust, 4)
    launches = steps * (3 * len(anchors) + len(reuse_layers))
    res["gpu_launches"] = launches
    # the dominant kernel of the Kascade prefill stack by total time: the
    # reuse-layer attention (24 launches per stack, one per reuse layer)
    pr_tf = f_reuse / (reuse_ms * 1e-3) / 1e12
    res["roofline"] = {"kernel": "k_prefill_fa2<reuse> (reuse layer)", "bound": "tensor",
                       "achieved": round(pr_tf, 1), "peak": tf_sust, "unit": "TFLOP/s",
                       "frac": round(pr_tf / tf_sust, 4), "traffic": TRAFFIC["k_prefill_fa2_reuse"],
                       "algorithmic_flops": int(f_reuse), "peak_source": src + " (sustained)"}
    del outs
    torch.cuda.empty_cache()
    clocks.begin()
    res["e2e"] = prefill_e2e(K, w, qs, ks, vs, anchors, ws, stream, steps, 1, world, dev)
    clocks.end()
    res["e2e"]["dense_ms_per_stack"] = res["dense_ms_per_stack"]
    rank = int(os.environ.get("RANK", "0"))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = time_oracle_prefill(w, [(qs[0], ks[0], vs[0]), (qs[1], ks[1], vs[1])],
                                                  n_units=2 * (os.cpu_count() or 1))
    del qs, ks, vs
    torch.cuda.empty_cache()
    return res, launches, ms_k, (anchor_ms, f_anchor, reuse_ms, f_reuse, tf_sust, src)


def time_anchor_layers(K, w, qs, ks, vs, ws, stream, reps, fused):
    """Mean CUDA-event time (us) of one anchor decode layer, taken over the
    workload's anchor layers in turn (each layer's K/V exceeds L2), with the
    two-kernel kascade_anchor_decode or the fused kascade_anchor_decode_fused."""
    import torch
    anchors = list(w.anchors)
    idx = torch.empty(w.batch, w.n_q_heads, w.topk, dtype=torch.int32, device=qs[0].device)
    out = torch.empty_like(qs[0])
    for a_ in anchors[:2]:
        K.anchor_decode(qs[a_], ks[a_], vs[a_], w.topk, out=out, idx=idx, ws=ws, fused=fused)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    n = 0
    for _ in range(reps):
        for a_ in anchors:
            K.anchor_decode(qs[a_], ks[a_], vs[a_], w.topk, out=out, idx=idx, ws=ws, fused=fused)
            n += 1
    e1.record(stream)
    torch.cuda.synchronize()
    assert ws.device_error() == K.OK
    return 1e3 * e0.elapsed_time(e1) / n


def fused_anchor_block(K, w, qs, ks, vs, ws, stream, reps, dense_us):
    """The anchor decode layer alone, two-kernel against fused (NEXT #2)."""
    two = time_anchor_layers(K, w, qs, ks, vs, ws, stream, reps, False)
    fused = time_anchor_layers(K, w, qs, ks, vs, ws, stream, reps, True)
    return {"anchor_layer_us_two_kernel": round(two, 2), "anchor_layer_us_fused": round(fused, 2),
            "fused_over_two_kernel": round(fused / two, 3),
            "anchor_over_dense_layer": round(two / dense_us, 3),
            "note": "kascade_anchor_decode (attention with logit spill, then Top-k) against "
                    "kascade_anchor_decode_fused (sample bracket, attention filing candidate "
                    "lists, selection from the lists); identical outputs"}


def stacked_layers(w, dev):
    """The workload's layers stacked into [L, ...] tensors (a step's host
    copies are then single transfers)."""
    import torch
    from long_context_anchor_gb300.workloads import layers as gen_layers
    B, Hq, Hkv, N, d, L = w.batch, w.n_q_heads, w.n_kv_heads, w.kv_len, w.head_dim, w.n_layers
    q_all = torch.empty(L, B, Hq, d, dtype=torch.bfloat16, device=dev)
    k_all = torch.empty(L, B, Hkv, N, d, dtype=torch.bfloat16, device=dev)
    v_all = torch.empty(L, B, Hkv, N, d, dtype=torch.bfloat16, device=dev)
    for l, (q, k, v) in enumerate(gen_layers(w, device=dev)):
        q_all[l].copy_(q)
        k_all[l].copy_(k)
        v_all[l].copy_(v)
        del q, k, v
    return q_all, k_all, v_all


def run_decode_tiny(args, dev, world, stream):
    """The tiny fp32 decode stack used for bring-up (B=1, 2 layers: anchor then
    reuse, Hq=4 / Hkv=2, d=64, N=512, k=32): its time is informational (launch
    latency bound), against the library's own dense decode on the same inputs."""
    import torch
    from long_context_anchor_gb300 import configs
    from long_context_anchor_gb300 import kascade as K
    from long_context_anchor_gb300.workloads import make_layers
    w = configs.TINY_DECODE
    qs, ks, vs = make_layers(w, device=dev)
    outs = [torch.empty_like(q) for q in qs]
    ws = K.Workspace(dev)
    anchors = list(w.anchors)

    def timed(anch, steps):
        for _ in range(args.warmup):
            K.run_stack(K.DECODE, qs, ks, vs, w.topk, anch, outs=outs, ws=ws)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            K.run_stack(K.DECODE, qs, ks, vs, w.topk, anch, outs=outs, ws=ws)
        e1.record(stream)
        torch.cuda.synchronize()
        assert ws.device_error() == K.OK
        return max_over_ranks([e0.elapsed_time(e1) / steps], world, dev)[0]

    steps = max(10, args.steps)
    ms_k, ms_d = timed(anchors, steps), timed([], steps)
    return {"workload": w.name, "layers": w.n_layers, "dtype": w.dtype,
            "kascade_us_per_layer": round(1e3 * ms_k / w.n_layers, 2),
            "dense_us_per_layer": round(1e3 * ms_d / w.n_layers, 2),
            "note": "bring-up size: launch latency, not bandwidth, sets these times"}


def run_decode_long(args, dev, world, stream, clocks):
    """Decode stack of the gpt-oss-20b-like attention shape (24 layers, 64/8
    heads, d=64, B=4, N=131072, k=8192, anchors every 3rd): Kascade vs the
    library's own dense decode, per-layer CUDA events, union bytes, the
    reuse kernel's roofline, an end-to-end pass with host buffers and the
    oracle on a sample."""
    import torch
    import torch.distributed as dist
    from long_context_anchor_gb300 import configs
    from long_context_anchor_gb300 import kascade as K
    w = configs.GPTOSS_DECODE_128K
    L = w.n_layers
    q_all, k_all, v_all = stacked_layers(w, dev)
    qs, ks, vs = list(q_all), list(k_all), list(v_all)
    out_all = torch.empty_like(q_all)
    outs = list(out_all)
    idx_buf = torch.empty(w.batch, w.n_q_heads, w.topk, dtype=torch.int32, device=dev)
    ws = K.Workspace(dev)
    anchors = list(w.anchors)

    def timed(anch, steps, per_layer=False):
        # headline without events between layers (see run_ours); per-layer
        # breakdown from a separate pass
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(L + 1)] for _ in range(steps)]
        for row in evs:
            for e in row:
                e.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for st in range(steps):
            if per_layer:
                evs[st][0].record(stream)
            K.run_stack(K.DECODE, qs, ks, vs, w.topk, anch, outs=outs, idx_buf=idx_buf, ws=ws,
                        layer_events=evs[st][1:] if per_layer else None)
        t1.record(stream)
        torch.cuda.synchronize()
        per = ([[evs[st][l].elapsed_time(evs[st][l + 1]) for l in range(L)] for st in range(steps)]
               if per_layer else None)
        return t0.elapsed_time(t1), per

    for _ in range(args.warmup):
        K.run_stack(K.DECODE, qs, ks, vs, w.topk, anchors, outs=outs, idx_buf=idx_buf, ws=ws)
        K.run_stack(K.DECODE, qs, ks, vs, w.topk, [], outs=outs, idx_buf=idx_buf, ws=ws)
    torch.cuda.synchronize()
    assert ws.device_error() == K.OK
    clocks.begin()
    tot_k, _ = timed(anchors, args.steps)
    tot_d, _ = timed([], args.steps)
    clocks.end()
    tot_k, tot_d = max_over_ranks([tot_k, tot_d], world, dev)
    steps_pl = max(2, args.steps // 2)
    _, per_k = timed(anchors, steps_pl, per_layer=True)
    ms_k, ms_d = tot_k / args.steps, tot_d / args.steps
    reuse_layers = [l for l in range(L) if l not in anchors]
    anchor_ms = statistics.mean(per_k[st][l] for st in range(steps_pl) for l in anchors)
    reuse_ms = statistics.mean(per_k[st][l] for st in range(steps_pl) for l in reuse_layers)
    unions = []
    for a_ in anchors:
        _, ia = K.anchor_decode(qs[a_], ks[a_], vs[a_], w.topk, ws=ws)
        unions.append(union_rows(ia, w))
    dense_b, anchor_b, reuse_b = decode_bytes(w, unions)
    seg = []
    for i, a_ in enumerate(anchors):
        nxt = anchors[i + 1] if i + 1 < len(anchors) else L
        seg += [reuse_b[i]] * (nxt - a_ - 1)
    reuse_bytes = statistics.mean(seg)
    reuse_gbs = reuse_bytes / (reuse_ms * 1e-3) / 1e9
    hbm_peak, _, src = load_peaks()
    res = {
        "workload": w.name, "layers": L, "batch": w.batch, "q_heads": w.n_q_heads,
        "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "kv_len": w.kv_len, "topk": w.topk,
        "anchors": anchors,
        "kascade_us_per_layer": round(1e3 * ms_k / L, 3),
        "dense_us_per_layer": round(1e3 * ms_d / L, 3),
        "speedup_vs_own_dense": round(ms_d / ms_k, 3),
        "anchor_layer_us": round(1e3 * anchor_ms, 3), "reuse_layer_us": round(1e3 * reuse_ms, 3),
        "reuse_hbm_gbs": round(reuse_gbs, 1), "reuse_frac_of_copy": round(reuse_gbs / hbm_peak, 4),
        "dense_hbm_gbs": round(dense_b / (ms_d / L * 1e-3) / 1e9, 1),
        "reuse_union_rows_per_layer": int(statistics.mean(unions)),
        "peak_hbm_gbs": hbm_peak, "peak_source": src,
        # the reuse-layer union gather: 16 of the 24 launches' layers, the
        # largest share of the Kascade stack's time
        "roofline": {"kernel": "k_decode_union_bf16 (reuse layer)", "bound": "hbm",
                     "achieved": round(reuse_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(reuse_gbs / hbm_peak, 4),
                     "frac_of_nominal_8tbs": round(reuse_gbs / NOMINAL_HBM_GBS, 4),
                     "traffic": TRAFFIC.get("k_decode_union_bf16_long"),
                     "algorithmic_bytes": int(reuse_bytes), "peak_source": src},
    }
    launches = args.steps * (3 * len(anchors) + len(reuse_layers))
    res["gpu_launches"] = launches
    clocks.begin()
    res["e2e"] = decode_e2e(K, w, q_all, k_all, v_all, out_all, anchors, idx_buf, ws, stream,
                            args.steps, args.warmup, world, dev)
    res["fused_anchor"] = fused_anchor_block(K, w, qs, ks, vs, ws, stream, max(2, args.steps // 4),
                                             1e3 * ms_d / L)
    clocks.end()
    rank = int(os.environ.get("RANK", "0"))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        lay01 = [(qs[0], ks[0], vs[0]), (qs[1], ks[1], vs[1])]
        res["cpu_baseline"] = time_oracle(w, lay01, n_groups=os.cpu_count() or 1, reps=1)
    del qs, ks, vs, outs, q_all, k_all, v_all, out_all
    torch.cuda.empty_cache()
    return res, launches


def run_ours(args):
    import torch
    import torch.distributed as dist
    from long_context_anchor_gb300 import configs
    from long_context_anchor_gb300 import kascade as K

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    w = configs.LLAMA8B_DECODE_32K
    L, B, Hq, Hkv, N, d = w.n_layers, w.batch, w.n_q_heads, w.n_kv_heads, w.kv_len, w.head_dim
    # Inputs resident in HBM, stacked so a step's host copies are single transfers.
    q_all, k_all, v_all = stacked_layers(w, dev)
    qs, ks, vs = list(q_all), list(k_all), list(v_all)
    out_all = torch.empty_like(q_all)
    outs = list(out_all)
    anchors = list(w.anchors)
    idx_buf = torch.empty(B, Hq, w.topk, dtype=torch.int32, device=dev)
    ws = K.Workspace(dev)
    stream = torch.cuda.current_stream()

    def stack(anch, events=None):
        K.run_stack(K.DECODE, qs, ks, vs, w.topk, anch, outs=outs, idx_buf=idx_buf, ws=ws,
                    layer_events=events)

    def timed(anch, steps, run=stack, per_layer=False):
        # The headline runs the stack without per-layer events: an event
        # between two layers' kernels would keep the next layer's kernels from
        # being scheduled early (programmatic dependent launch). The per-layer
        # breakdown comes from a separate pass with events.
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(L + 1)] for _ in range(steps)]
        for row in evs:
            for e in row:
                e.record(stream)        # materialise the event handles
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for s in range(steps):
            if per_layer:
                evs[s][0].record(stream)
                run(anch, evs[s][1:])
            else:
                run(anch)
        t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        total = t0.elapsed_time(t1)
        per = ([[evs[s][l].elapsed_time(evs[s][l + 1]) for l in range(L)] for s in range(steps)]
               if per_layer else None)
        return total, per

    for _ in range(args.warmup):
        stack(anchors)
        stack([])
    torch.cuda.synchronize()
    assert ws.device_error() == K.OK

    clocks = ClockSampler(local)
    clocks.start()
    clocks.begin()
    total_k, _ = timed(anchors, args.steps)
    total_d, _ = timed([], args.steps)
    clocks.end()
    total_k, total_d = max_over_ranks([total_k, total_d], world, dev)
    # per-layer breakdown (events between layers)
    steps_pl = max(2, args.steps // 2)
    _, pl_k = timed(anchors, steps_pl, per_layer=True)

    ms_step = total_k / args.steps
    ms_dense = total_d / args.steps
    anchor_ms = statistics.mean(pl_k[s][l] for s in range(steps_pl) for l in anchors)
    reuse_layers = [l for l in range(L) if l not in anchors]
    reuse_ms = statistics.mean(pl_k[s][l] for s in range(steps_pl) for l in reuse_layers)

    # Byte accounting from each anchor's own sets (outside the timed region).
    unions = []
    for a in anchors:
        _, ia = K.anchor_decode(qs[a], ks[a], vs[a], w.topk, ws=ws)
        unions.append(union_rows(ia, w))
    dense_b, anchor_b, reuse_b = decode_bytes(w, unions)
    seg_reuse = []
    for i, a in enumerate(anchors):
        nxt = anchors[i + 1] if i + 1 < len(anchors) else L
        seg_reuse += [reuse_b[i]] * (nxt - a - 1)
    reuse_bytes_mean = statistics.mean(seg_reuse)
    anchor_bytes_mean = statistics.mean(anchor_b)
    hbm_peak, tf_peak, peak_src = load_peaks()
    reuse_gbs = reuse_bytes_mean / (reuse_ms * 1e-3) / 1e9
    anchor_gbs = anchor_bytes_mean / (anchor_ms * 1e-3) / 1e9
    dense_gbs = dense_b / (ms_dense / L * 1e-3) / 1e9
    stack_bytes = sum(anchor_b) + sum(seg_reuse)
    launches_per_step = 3 * len(anchors) + len(reuse_layers)

    result = {
        "metric": METRIC, "value": round(1e3 * ms_step / L, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "layers": L, "batch": B, "q_heads": Hq, "kv_heads": Hkv,
                   "head_dim": d, "kv_len": N, "topk": w.topk, "anchors": anchors,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "no flush: each layer's K/V (1.07 GB) is distinct and exceeds L2"},
        "decode": {"kascade_us_per_layer": round(1e3 * ms_step / L, 3),
                   "anchor_layer_us": round(1e3 * anchor_ms, 3),
                   "reuse_layer_us": round(1e3 * reuse_ms, 3),
                   "dense_us_per_layer": round(1e3 * ms_dense / L, 3),
                   "speedup_vs_own_dense": round(ms_dense / ms_step, 3),
                   "stack_hbm_gbs": round(stack_bytes / (ms_step * 1e-3) / 1e9, 1),
                   "reuse_hbm_gbs": round(reuse_gbs, 1), "anchor_hbm_gbs": round(anchor_gbs, 1),
                   "dense_hbm_gbs": round(dense_gbs, 1),
                   "reuse_union_rows_per_layer": int(statistics.mean(unions)),
                   "reuse_bytes_per_layer": int(reuse_bytes_mean),
                   "anchor_bytes_per_layer": int(anchor_bytes_mean),
                   "dense_bytes_per_layer": int(dense_b),
                   "peak_hbm_gbs": hbm_peak, "peak_source": peak_src},
        "gpu_launches": launches_per_step * args.steps,
    }
    # Dominant kernel of the headline decode step: the reuse-layer union
    # gather (24 launches per step, 1.9 ms of the 3.6 ms step; the anchor
    # layers' dense read with the logit spill takes 8 launches).
    result["roofline"] = {"kernel": "k_decode_union_bf16 (reuse layer)", "bound": "hbm",
                          "achieved": round(reuse_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                          "frac": round(reuse_gbs / hbm_peak, 4),
                          "frac_of_nominal_8tbs": round(reuse_gbs / NOMINAL_HBM_GBS, 4),
                          "traffic": TRAFFIC["k_decode_union_bf16"],
                          "algorithmic_bytes": int(reuse_bytes_mean),
                          "peak_source": peak_src}
    result["roofline_decode_anchor_layer"] = {
        "kernel": "anchor layer (k_decode_dense_bf16 with logit spill + k_topk + plan)",
        "bound": "hbm", "achieved": round(anchor_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
        "frac": round(anchor_gbs / hbm_peak, 4), "traffic": None,
        "algorithmic_bytes": int(anchor_bytes_mean), "peak_source": peak_src}

    clocks.begin()
    result["e2e"] = decode_e2e(K, w, q_all, k_all, v_all, out_all, anchors, idx_buf, ws, stream,
                               args.steps, args.warmup, world, dev)
    result["decode"]["fused_anchor"] = fused_anchor_block(K, w, qs, ks, vs, ws, stream,
                                                          max(2, args.steps // 4),
                                                          1e3 * ms_dense / L)
    clocks.end()
    # GQA-pooled index sets (one per KV head) on the same resident inputs.
    if not args.no_pooled:
        idx_pool = torch.empty(B, Hkv, w.topk, dtype=torch.int32, device=dev)

        def stack_pooled(anch, events=None):
            K.run_stack(K.DECODE, qs, ks, vs, w.topk, anch, outs=outs, idx_buf=idx_pool, ws=ws,
                        layer_events=events, pooled=True)

        for _ in range(args.warmup):
            stack_pooled(anchors)
        torch.cuda.synchronize()
        assert ws.device_error() == K.OK
        clocks.begin()
        total_p, _ = timed(anchors, args.steps, stack_pooled)
        clocks.end()
        total_p = max_over_ranks([total_p], world, dev)[0]
        _, pl_p = timed(anchors, steps_pl, stack_pooled, per_layer=True)
        ms_p = total_p / args.steps
        anchor_p = statistics.mean(pl_p[s][l] for s in range(steps_pl) for l in anchors)
        reuse_p = statistics.mean(pl_p[s][l] for s in range(steps_pl) for l in reuse_layers)
        pa_b, pr_b = pooled_decode_bytes(w)
        pr_gbs = pr_b / (reuse_p * 1e-3) / 1e9
        result["decode_pooled"] = {
            "index_sets": "one per (sequence, KV head): group sums of softmax weights",
            "kascade_us_per_layer": round(1e3 * ms_p / L, 3),
            "anchor_layer_us": round(1e3 * anchor_p, 3),
            "reuse_layer_us": round(1e3 * reuse_p, 3),
            "speedup_vs_own_dense": round(ms_dense / ms_p, 3),
            "reuse_hbm_gbs": round(pr_gbs, 1), "reuse_frac_of_copy": round(pr_gbs / hbm_peak, 4),
            "reuse_bytes_per_layer": int(pr_b), "anchor_bytes_per_layer": int(pa_b),
            "anchor_hbm_gbs": round(pa_b / (anchor_p * 1e-3) / 1e9, 1)}
        # anchor: attention (which also leaves the row statistics), pooled
        # weights, Top-k; reuse: one gather
        result["gpu_launches_decode_pooled"] = args.steps * (3 * len(anchors) + len(reuse_layers))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        lay01 = [(qs[0], ks[0], vs[0]), (qs[1], ks[1], vs[1])]
        result["cpu_baseline"] = time_oracle(w, lay01, n_groups=os.cpu_count() or 1, reps=2)
    del qs, ks, vs, outs, q_all, k_all, v_all, out_all, idx_buf, ws
    torch.cuda.empty_cache()
    result["decode_tiny"] = run_decode_tiny(args, dev, world, stream)
    # Prefill stack: Llama-3.1-8B shape at N = 16384.
    if not args.no_prefill:
        pre, pre_launches, pre_ms, _ = run_prefill(args, dev, world, stream, clocks)
        result["prefill"] = pre
        result["gpu_launches_prefill"] = pre_launches
        result["ms_per_step_prefill"] = round(pre_ms, 3)
    if not args.no_long_decode:
        long_res, long_launches = run_decode_long(args, dev, world, stream, clocks)
        result["decode_long"] = long_res
        result["gpu_launches_decode_long"] = long_launches
    # Schedule sweep: DP anchors from calibration, then decode B16 and
    # prefill at three lengths against the library's own dense kernels.
    if not args.no_sweep:
        result["sweep"] = run_sweep(args, clocks=clocks, world=world, dev=dev)
    result["clocks"] = clocks.stop()
    if world > 1:
        dist.destroy_process_group()
    return result if rank == 0 else None


def run_reference(args):
    """The CPU oracle as the reference arm, on a bounded sample per step."""
    import torch
    from long_context_anchor_gb300 import configs
    from long_context_anchor_gb300.workloads import make_layers
    rank, world, local = dist_env()
    if rank != 0:
        return None
    w = configs.LLAMA8B_DECODE_32K
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    qs, ks, vs = make_layers(w.with_(n_layers=2), device=dev)
    lay01 = [(qs[0], ks[0], vs[0]), (qs[1], ks[1], vs[1])]
    n = os.cpu_count() or 1
    for _ in range(args.warmup):
        time_oracle(w, lay01, n_groups=n, reps=1)
    vals = [time_oracle(w, lay01, n_groups=n, reps=1) for _ in range(args.steps)]
    us = statistics.mean(v["value"] for v in vals)
    cb = dict(vals[0])
    cb["value"] = us
    return {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(us * w.n_layers / 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "layers": w.n_layers, "batch": w.batch,
                       "kv_len": w.kv_len, "topk": w.topk, "anchors": list(w.anchors)},
            "cpu_baseline": cb,
            "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_sweep(args, clocks=None, world=1, dev=None):
    """Schedule sweep (the 32-layer 8B shape): the DP picks six anchors from
    calibration on four synthetic sequences (overlap similarity, and the
    mass-recall similarity beside it), then the decode stack at batch 16 and
    the prefill stack at N = 4096, 16384 and 65536 run with those anchors
    against the library's own dense kernels on the same inputs."""
    import torch
    from long_context_anchor_gb300 import configs
    from long_context_anchor_gb300 import kascade as K
    from long_context_anchor_gb300.schedule_file import objective as schedule_objective
    from long_context_anchor_gb300.schedule_file import save_schedule
    from long_context_anchor_gb300.workloads import make_layers
    dev = dev if dev is not None else torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    res = {"data": "synthetic", "dtype": "bf16"}
    # 1. calibration + DP
    wc = configs.SWEEP_CALIBRATION
    qs, ks, vs = make_layers(wc, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    sim, _ = K.calibrate(qs, ks, vs, wc.topk)
    t_cal = time.perf_counter() - t0
    m = configs.SWEEP_N_ANCHORS
    anchors, obj = K.schedule_anchors(sim, m)
    L = wc.n_layers
    uniform = list(range(0, L, L // m))[:m]
    # the same DP on the attention-mass-recall similarity
    t0 = time.perf_counter()
    rsim, _ = K.calibrate(qs, ks, vs, wc.topk, similarity="recall")
    t_rcal = time.perf_counter() - t0
    r_anchors, r_obj = K.schedule_anchors(rsim, m)
    res["calibration"] = {"workload": wc.name, "seconds": round(t_cal, 3), "anchors": anchors,
                          "objective": round(obj, 4),
                          "uniform_anchors": uniform,
                          "uniform_objective": round(schedule_objective(uniform, sim), 4),
                          "sim_adjacent_mean": round(float(np.mean([sim[i][i + 1] for i in range(L - 1)])), 4)}
    # mean share of each layer's exact attention mass kept by the set it
    # reuses, under each schedule (the recall objective / L)
    res["calibration_recall"] = {
        "seconds": round(t_rcal, 3), "anchors": r_anchors, "objective": round(r_obj, 4),
        "mass_kept_recall_anchors": round(r_obj / L, 4),
        "mass_kept_overlap_anchors": round(schedule_objective(anchors, rsim) / L, 4),
        "mass_kept_uniform_anchors": round(schedule_objective(uniform, rsim) / L, 4),
        "mass_kept_own_topk_mean": round(float(np.mean([rsim[l][l] for l in range(L)])), 4)}
    if args.save_schedule:
        meta = {"workload": wc.name, "topk": wc.topk, "batch": wc.batch, "kv_len": wc.kv_len,
                "n_q_heads": wc.n_q_heads, "n_kv_heads": wc.n_kv_heads, "data": "synthetic"}
        save_schedule(args.save_schedule, anchors, sim, "overlap", meta)
        root, ext = os.path.splitext(args.save_schedule)
        save_schedule(root + "_recall" + (ext or ".json"), r_anchors, rsim, "recall", meta)
        res["schedule_files"] = [args.save_schedule, root + "_recall" + (ext or ".json")]
    del qs, ks, vs
    torch.cuda.empty_cache()

    def time_stack(mode, qs, ks, vs, topk, anch, steps, warm):
        outs = [torch.empty_like(q) for q in qs]
        ws = K.Workspace(dev)
        for _ in range(warm):
            K.run_stack(mode, qs, ks, vs, topk, anch, outs=outs, ws=ws)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if clocks is not None:
            clocks.begin()
        e0.record(stream)
        for _ in range(steps):
            K.run_stack(mode, qs, ks, vs, topk, anch, outs=outs, ws=ws)
        e1.record(stream)
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.end()
        assert ws.device_error() == K.OK
        return max_over_ranks([e0.elapsed_time(e1) / steps], world, dev)[0]

    # 2. decode, batch 16, N = 32768
    wd = configs.SWEEP_DECODE
    qs, ks, vs = make_layers(wd, device=dev)
    warm = max(3, args.warmup)
    ms_k = time_stack(K.DECODE, qs, ks, vs, wd.topk, anchors, args.steps, warm)
    ms_d = time_stack(K.DECODE, qs, ks, vs, wd.topk, [], args.steps, warm)
    res["decode"] = {"workload": wd.name, "anchors": anchors, "steps": args.steps,
                     "kascade_us_per_layer": round(1e3 * ms_k / wd.n_layers, 2),
                     "dense_us_per_layer": round(1e3 * ms_d / wd.n_layers, 2),
                     "speedup_vs_own_dense": round(ms_d / ms_k, 3)}
    del qs, ks, vs
    torch.cuda.empty_cache()
    # 3. prefill at three lengths (fewer steps as N grows)
    res["prefill"] = []
    for n in configs.SWEEP_PREFILL_LENGTHS:
        wp = configs.sweep_prefill(n)
        qs, ks, vs = make_layers(wp, device=dev)
        steps = max(2, args.steps * 4096 // (4 * n))
        ms_k = time_stack(K.PREFILL, qs, ks, vs, wp.topk, anchors, steps, 1)
        ms_d = time_stack(K.PREFILL, qs, ks, vs, wp.topk, [], steps, 1)
        f_dense, f_anchor, f_reuse = prefill_flops(wp)
        flops_k = len(anchors) * f_anchor + (wp.n_layers - len(anchors)) * f_reuse
        res["prefill"].append({"workload": wp.name, "steps": steps,
                               "kascade_ms_per_stack": round(ms_k, 2),
                               "dense_ms_per_stack": round(ms_d, 2),
                               "speedup_vs_own_dense": round(ms_d / ms_k, 3),
                               "kascade_tflops": round(flops_k / (ms_k * 1e-3) / 1e12, 1),
                               "dense_tflops": round(wp.n_layers * f_dense / (ms_d * 1e-3) / 1e12, 1)})
        del qs, ks, vs
        torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-long-decode", action="store_true",
                    help="skip the gpt-oss-20b-like decode stack (N=131072, d=64)")
    ap.add_argument("--no-pooled", action="store_true",
                    help="skip the decode stack with GQA-pooled index sets")
    ap.add_argument("--sweep", action="store_true",
                    help="only the schedule sweep: DP anchors from calibration, decode and "
                         "prefill vs dense")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the schedule sweep leg of the default run")
    ap.add_argument("--save-schedule", default="",
                    help="with --sweep: write the DP schedules (overlap, and recall beside it) as JSON")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.sweep:
        res = {"impl": "ours", "mode": "sweep", "metric": METRIC}
        res.update(run_sweep(args))
    else:
        res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
