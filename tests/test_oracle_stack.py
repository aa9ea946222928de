"""Pins for oracle/stack.py: reuse layers read exactly the most recent
anchor's index sets; anchors output dense attention; layers before the first
anchor run dense."""
import numpy as np

from oracle import attention as A
from oracle.stack import run_stack


def _layers(rng, L, mode, B=1, Hq=4, Hkv=2, N=64, d=8):
    out = []
    for _ in range(L):
        if mode == "decode":
            q = rng.standard_normal((B, Hq, d))
        else:
            q = rng.standard_normal((B, Hq, N, d))
        out.append((q, rng.standard_normal((B, Hkv, N, d)), rng.standard_normal((B, Hkv, N, d))))
    return out


def test_decode_stack_reads_anchor_sets():
    rng = np.random.default_rng(0)
    layers = _layers(rng, 7, "decode")
    outs, read, written = run_stack("decode", layers, 8, [1, 4])
    # layer 0 precedes the first anchor: dense, nothing read
    np.testing.assert_array_equal(outs[0], A.dense_decode(*layers[0])[0])
    assert read[0] is None and written[0] is None
    for layer in (2, 3):
        assert read[layer] is written[1]
    for layer in (5, 6):
        assert read[layer] is written[4]
    np.testing.assert_array_equal(outs[4], A.anchor_decode(*layers[4], 8)[0])
    np.testing.assert_array_equal(outs[5], A.sparse_decode(*layers[5], written[4]))
    # the set layer 4 wrote is layer 4's own Top-k
    np.testing.assert_array_equal(written[4], A.anchor_decode(*layers[4], 8)[1])


def test_prefill_stack_reads_anchor_sets():
    rng = np.random.default_rng(1)
    layers = _layers(rng, 3, "prefill", N=200)
    outs, read, written = run_stack("prefill", layers, 16, [0])
    assert read[1] is written[0] and read[2] is written[0]
    np.testing.assert_array_equal(outs[2], A.sparse_prefill(*layers[2], written[0]))


def test_pooled_stacks_hold_per_kv_head_sets():
    rng = np.random.default_rng(2)
    layers = _layers(rng, 4, "decode")
    outs, read, written = run_stack("decode", layers, 8, [0, 2], pooled=True)
    assert written[0].shape == (1, 2, 8)     # [B, Hkv, k]
    assert read[1] is written[0] and read[3] is written[2]
    np.testing.assert_array_equal(outs[3], A.sparse_decode_pooled(*layers[3], written[2]))
    np.testing.assert_array_equal(written[2], A.anchor_decode_pooled(*layers[2], 8)[1])
    layers = _layers(rng, 2, "prefill", N=200)
    outs, read, written = run_stack("prefill", layers, 16, [0], pooled=True)
    assert written[0].shape == (1, 2, 2, 16)  # [B, Hkv, nT, k]
    np.testing.assert_array_equal(outs[1], A.sparse_prefill_pooled(*layers[1], written[0]))
