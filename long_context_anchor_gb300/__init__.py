"""Kascade head-aware Top-k sparse attention with cross-layer index reuse, for GB300.

The compute path is the in-tree CUDA library ``libkascade.so`` (see
``include/kascade.h``); ``long_context_anchor_gb300.kascade`` is its Python
binding. ``workloads`` and ``configs`` draw synthetic inputs. Importing this
package does not load the library; ``from long_context_anchor_gb300 import
kascade`` does, and fails loudly if it has not been built.
"""
