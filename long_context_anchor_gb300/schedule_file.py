"""Anchor schedules on disk.

Kascade picks its anchor layers offline, by a dynamic programme over the
cross-layer similarity of Top-k sets measured on calibration data, and then
uses that fixed list at inference (euno.news summary, Key Contributions and
Methodology 4). This module stores such a schedule as JSON: the anchor list,
the similarity matrix it was chosen from, which similarity that was
("overlap" or "recall"), the DP objective, and free-form metadata (the
calibration shape, the Top-k size). Loading checks the file against itself:
the anchors are ascending layer indices and the stored objective equals the
one the anchors reach on the stored matrix, so a schedule cannot drift from
the matrix it claims to come from.

    F(A) = sum over layers l >= A[0] of sim[a(l)][l], a(l) = max{a in A : a <= l}

Layers before the first anchor run dense and add no term.
"""
import json
import math
import os
import tempfile
from typing import Any, Dict, Optional, Sequence

FORMAT = "kascade-anchor-schedule/1"
SIMILARITIES = ("overlap", "recall")


class ScheduleError(ValueError):
    pass


def check_anchors(anchors: Sequence[int], n_layers: int) -> list:
    """Anchors as a list of ints, strictly ascending, each in [0, n_layers)."""
    out = []
    for a in anchors:
        if isinstance(a, bool) or not isinstance(a, int):
            raise ScheduleError("anchors must be integers, got %r" % (a,))
        if not 0 <= a < n_layers:
            raise ScheduleError("anchor %d outside [0, %d)" % (a, n_layers))
        if out and a <= out[-1]:
            raise ScheduleError("anchors must be strictly ascending: %r" % (list(anchors),))
        out.append(a)
    if not out:
        raise ScheduleError("a schedule needs at least one anchor")
    return out


def check_matrix(sim) -> list:
    """A square matrix of finite floats, as a list of lists."""
    rows = [list(r) for r in sim]
    L = len(rows)
    if L == 0 or any(len(r) != L for r in rows):
        raise ScheduleError("similarity must be a non-empty square matrix")
    out = []
    for r in rows:
        vals = [float(x) for x in r]
        if not all(math.isfinite(x) for x in vals):
            raise ScheduleError("similarity entries must be finite")
        out.append(vals)
    return out


def objective(anchors: Sequence[int], sim) -> float:
    """F(A): each layer from the first anchor on scores its most recent anchor's row."""
    L = len(sim)
    total, cur, nxt = 0.0, None, 0
    for layer in range(L):
        if nxt < len(anchors) and anchors[nxt] == layer:
            cur = layer
            nxt += 1
        if cur is not None:
            total += float(sim[cur][layer])
    return total


def save_schedule(path: str, anchors: Sequence[int], sim, similarity: str = "overlap",
                  meta: Optional[Dict[str, Any]] = None) -> Dict[str, Any]:
    """Write a schedule (atomically: a temporary file renamed over `path`); returns it."""
    if similarity not in SIMILARITIES:
        raise ScheduleError("similarity must be one of %s" % (SIMILARITIES,))
    m = check_matrix(sim)
    a = check_anchors(anchors, len(m))
    doc = {"format": FORMAT, "n_layers": len(m), "anchors": a, "similarity": similarity,
           "objective": objective(a, m), "sim": m, "meta": dict(meta or {})}
    text = json.dumps(doc, indent=1, sort_keys=True)
    d = os.path.dirname(os.path.abspath(path))
    fd, tmp = tempfile.mkstemp(prefix=".schedule-", suffix=".json", dir=d)
    try:
        with os.fdopen(fd, "w") as f:
            f.write(text + "\n")
        os.replace(tmp, path)
    except BaseException:
        if os.path.exists(tmp):
            os.unlink(tmp)
        raise
    return doc


def load_schedule(path: str) -> Dict[str, Any]:
    """Read and check a schedule written by save_schedule."""
    with open(path) as f:
        doc = json.load(f)
    if not isinstance(doc, dict) or doc.get("format") != FORMAT:
        raise ScheduleError("%s: not a %s file" % (path, FORMAT))
    m = check_matrix(doc.get("sim", []))
    if doc.get("n_layers") != len(m):
        raise ScheduleError("n_layers %r does not match the %d x %d matrix"
                            % (doc.get("n_layers"), len(m), len(m)))
    a = check_anchors(doc.get("anchors", []), len(m))
    if doc.get("similarity") not in SIMILARITIES:
        raise ScheduleError("unknown similarity %r" % (doc.get("similarity"),))
    f_a = objective(a, m)
    stored = doc.get("objective")
    if not isinstance(stored, (int, float)) or abs(float(stored) - f_a) > 1e-9 * max(1.0, abs(f_a)):
        raise ScheduleError("stored objective %r differs from F(A) = %r" % (stored, f_a))
    doc["anchors"], doc["sim"], doc["objective"] = a, m, f_a
    doc.setdefault("meta", {})
    return doc
