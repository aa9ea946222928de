"""Shared checks for the GPU parity tests (comparison logic only; no method arithmetic)."""
import numpy as np
import torch

# Tolerances: attention outputs max-abs 2e-2 and mean-abs 2e-3 against the
# float64 oracle; an index that differs from the oracle's set must score
# within 1e-3 of the oracle's k-th score.
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
INDEX_SCORE_TOL = 1e-3


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_out(got, ref, max_abs=OUT_MAX_ABS, mean_abs=OUT_MEAN_ABS, what="out"):
    g = f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.isfinite(g).all(), what
    err = np.abs(g - r)
    assert err.max() <= max_abs, (what, float(err.max()))
    assert err.mean() <= mean_abs, (what, float(err.mean()))
    return float(err.max()), float(err.mean())


def check_index_set(got_row, ref_scores, k, tol=INDEX_SCORE_TOL, what="idx"):
    """got_row: selected positions (ascending, distinct); ref_scores: oracle scores of the row."""
    got = np.asarray(got_row, dtype=np.int64)
    got = got[got >= 0]
    k = min(k, ref_scores.shape[0])
    assert got.shape[0] == k, (what, got.shape[0], k)
    assert (np.diff(got) > 0).all(), (what, "not strictly ascending")
    assert got.min() >= 0 and got.max() < ref_scores.shape[0], what
    kth = np.sort(ref_scores)[::-1][k - 1]
    ref_sel = set(np.lexsort((np.arange(ref_scores.shape[0]), -ref_scores))[:k].tolist())
    diff = set(got.tolist()) ^ ref_sel
    bad = [j for j in diff if abs(ref_scores[j] - kth) > tol]
    assert not bad, (what, len(diff), bad[:5], kth)
    return len(diff)
