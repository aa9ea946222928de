"""CPU oracle for Kascade head-aware Top-k sparse attention with cross-layer reuse.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The library (``long_context_anchor_gb300``) never calls it and has no
CPU fallback.

Everything here is plain numpy in float64, evaluated on host copies of the
same (bf16- or fp32-valued) inputs the GPU path receives. It follows the
method as the Kascade pages state it ("Kascade: A Practical Sparse Attention
Method for Long-Context LLM Inference"; euno.news summary, sections *Key
Contributions* and *Methodology*; opentrain.ai page, *Abstract*):

* anchor layers compute attention exactly, then an exact per-head Top-k of key
  indices (Methodology 2, 5; Abstract);
* reuse layers recompute attention with their own q, K, V, softmax restricted
  to the saved set (Methodology 3);
* prefill works per query tile (Abstract: "tile-level operations"), one index
  set per (head, 128-row tile) ranked by the tile's summed post-softmax
  weights;
* anchors are chosen by a dynamic programme maximising cross-layer Top-k
  overlap (Key Contributions; Methodology 4);
* optionally (GQA-pooled sets) one set per (sequence, KV head), ranked by
  the sum of the group's query heads' post-softmax (or tile) weights: a
  reading for GQA models, whose head granularity the pages leave open.

Modules: ``attention`` (dense / sparse decode and prefill), ``topk`` (the
selection rule), ``schedule`` (overlap similarity and the anchor DP),
``stack`` (the layer-stack driver). Pins live in ``tests/test_oracle_*.py``.
No function here is "parity unpinned".
"""
