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


# Tile weights (prefill) and pooled weights are sums of probabilities; the
# kernel's fp32 logits are within 1e-3 of the oracle's, which moves exp(s) by
# at most ~1e-3 relative, so they are compared with a relative 2e-3.
WEIGHT_REL = 2e-3
# An end-to-end set may differ from the oracle's only on near-ties: every
# differing position must pass the score tolerance above, and there may be
# at most 1% of k of them (at least 2). At the kernels' actual fp32 error
# (~1e-5 relative) the expected number is well below one per row.
MAX_DIFF_FRAC = 0.01


def log_w(w):
    """log of non-negative weights (0 -> -inf), the scale near-ties of
    probability-like scores are judged on."""
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(w, dtype=np.float64))


def check_weights(got, ref, rel=WEIGHT_REL, what="weights"):
    g = f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape and np.isfinite(g).all(), (what, g.shape, r.shape)
    err = np.abs(g - r)
    assert (err <= rel * np.abs(r) + 1e-12).all(), (what, float((err / (np.abs(r) + 1e-30)).max()))
    return float((err / (np.abs(r) + 1e-30)).max())


def packed_tile(w_row, t, n, tile=128):
    """Tile t's weights (L_t of them) inside one packed (sequence, head) row."""
    off = (tile // 2) * t * (t + 1)
    return w_row[off:off + min(n, tile * (t + 1))]


def check_index_set(got_row, ref_scores, k, tol=INDEX_SCORE_TOL, what="idx",
                    max_diff_frac=MAX_DIFF_FRAC):
    """got_row: selected positions (ascending, distinct); ref_scores: oracle scores of the row
    (logits, or log-weights for probability-like scores)."""
    got = np.asarray(got_row, dtype=np.int64)
    got = got[got >= 0]
    k = min(k, ref_scores.shape[0])
    assert got.shape[0] == k, (what, got.shape[0], k)
    assert (np.diff(got) > 0).all(), (what, "not strictly ascending")
    assert got.min() >= 0 and got.max() < ref_scores.shape[0], what
    kth = np.sort(ref_scores)[::-1][k - 1]
    ref_sel = set(np.lexsort((np.arange(ref_scores.shape[0]), -ref_scores))[:k].tolist())
    diff = set(got.tolist()) ^ ref_sel
    bad = [j for j in diff if not abs(ref_scores[j] - kth) <= tol]
    assert not bad, (what, len(diff), bad[:5], kth)
    # each swap puts one position in and one out
    assert len(diff) // 2 <= max(2, int(max_diff_frac * k)), (what, "too many swaps", len(diff))
    return len(diff)


def check_topk_exact(got_row, scores_row, k, what="topk"):
    """Bit-exact Top-k: the kernel's set on its own fp32 scores equals the
    oracle rule applied to the identical fp32 array."""
    from oracle.topk import topk_indices
    got = np.asarray(got_row, dtype=np.int64)
    k = min(k, np.shape(scores_row)[0])
    exp = topk_indices(np.asarray(scores_row, dtype=np.float32), k)
    assert got[:k].tolist() == exp.tolist(), (what, "set differs from the rule on identical scores")
    assert (got[k:] == -1).all(), (what, "padding")
