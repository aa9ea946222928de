"""Exact Top-k selection rule (oracle).

Kascade selects "exact top-k attention indices" per head (euno.news summary,
Key Contributions "Cross-layer Top-k reuse" and "Head-aware selection";
Methodology 2 and 5). The pages fix neither tie-breaking nor output order;
the readings used here are:

* order: score descending, then index ascending (lower index wins a tie);
* -0.0 and +0.0 are equal; -inf is a valid score and ranks last;
* NaN is rejected as invalid input;
* the selected indices are returned sorted ascending;
* when k >= n every position is selected.
"""
import numpy as np


def topk_indices(scores, k: int) -> np.ndarray:
    """Indices of the min(k, n) largest scores under the rule above, ascending."""
    s = np.asarray(scores)
    if s.ndim != 1:
        raise ValueError("scores must be 1-D")
    if np.isnan(s).any():
        raise ValueError("NaN score")
    n = s.shape[0]
    k = min(int(k), n)
    if k <= 0:
        return np.zeros(0, dtype=np.int64)
    # lexsort: last key is primary. Primary = -score (so larger scores first;
    # -(-0.0) == -(+0.0) compares equal), secondary = index ascending.
    order = np.lexsort((np.arange(n), -s.astype(np.float64)))
    return np.sort(order[:k])


def kth_score(scores, k: int) -> float:
    """The k-th largest score (the selection threshold)."""
    s = np.sort(np.asarray(scores, dtype=np.float64))[::-1]
    return float(s[min(k, s.shape[0]) - 1])
