"""The five synthetic workloads the library is measured and checked on.

Shapes follow the attention of the models the Kascade pages evaluate
(Llama-3.1-8B: 32 query / 8 KV heads, head_dim 128; gpt-oss-20b-like:
64 query / 8 KV heads, head_dim 64). Seeds are 1000 + workload number.
"""
from .workloads import Workload

TINY_DECODE = Workload(
    name="tiny_decode_b1_hq4_hkv2_d64_n512_k32_f32", mode="decode", n_layers=2, batch=1,
    n_q_heads=4, n_kv_heads=2, head_dim=64, kv_len=512, topk=32, anchors=(0,),
    dtype="f32", n_plants=16, plant_strength=3.0, sink=False, rho=0.9, seed=1000)

LLAMA8B_DECODE_32K = Workload(
    name="llama8b_decode_b8_n32768_k4096", mode="decode", n_layers=32, batch=8,
    n_q_heads=32, n_kv_heads=8, head_dim=128, kv_len=32768, topk=4096,
    anchors=tuple(range(0, 32, 4)), dtype="bf16", n_plants=64, plant_strength=3.0,
    sink=True, rho=0.9, seed=1001)

LLAMA8B_PREFILL_16K = Workload(
    name="llama8b_prefill_n16384_k2048", mode="prefill", n_layers=32, batch=1,
    n_q_heads=32, n_kv_heads=8, head_dim=128, kv_len=16384, topk=2048,
    anchors=tuple(range(0, 32, 4)), dtype="bf16", n_plants=64, plant_strength=3.0,
    sink=True, rho=0.9, seed=1002)

GPTOSS_DECODE_128K = Workload(
    name="gptoss20b_decode_b4_n131072_k8192", mode="decode", n_layers=24, batch=4,
    n_q_heads=64, n_kv_heads=8, head_dim=64, kv_len=131072, topk=8192,
    anchors=tuple(range(0, 24, 3)), dtype="bf16", n_plants=128, plant_strength=3.0,
    sink=True, rho=0.85, seed=1003)

# Schedule sweep: calibration on 4 sequences with per-layer rho ~ U[0.7, 0.95],
# 6 anchors chosen by the DP, then evaluation at the lengths below. The
# evaluation inputs are fresh sequences (their own seeds) on the same
# per-layer rhos as the calibration (rho_seed).
SWEEP_CALIBRATION = Workload(
    name="llama8b_calibration_b4_n32768_k4096", mode="decode", n_layers=32, batch=4,
    n_q_heads=32, n_kv_heads=8, head_dim=128, kv_len=32768, topk=4096,
    anchors=tuple(range(32)), dtype="bf16", n_plants=64, plant_strength=3.0,
    sink=True, rho_range=(0.7, 0.95), seed=1004)
SWEEP_N_ANCHORS = 6
SWEEP_PREFILL_LENGTHS = (4096, 16384, 65536)
SWEEP_DECODE = SWEEP_CALIBRATION.with_(name="llama8b_decode_b16_n32768_k4096", batch=16,
                                       seed=2004, rho_seed=SWEEP_CALIBRATION.seed)


def sweep_prefill(n: int) -> Workload:
    """Sweep evaluation prefill at length n (k = n/8), 32 layers of the 8B shape."""
    return LLAMA8B_PREFILL_16K.with_(name="llama8b_prefill_n%d_k%d" % (n, n // 8), kv_len=n,
                                     topk=n // 8, rho_range=(0.7, 0.95), seed=3004 + n,
                                     rho_seed=SWEEP_CALIBRATION.seed)

ALL = [TINY_DECODE, LLAMA8B_DECODE_32K, LLAMA8B_PREFILL_16K, GPTOSS_DECODE_128K,
       SWEEP_CALIBRATION]
