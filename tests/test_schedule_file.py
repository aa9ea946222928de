"""Anchor schedule files: a round trip keeps the anchors, matrix and
objective; the stored objective equals the host DP's; malformed or
inconsistent files are refused. No GPU."""
import json

import numpy as np
import pytest

import __graft_entry__
from long_context_anchor_gb300 import schedule_file as SF


@pytest.fixture(scope="module")
def K():
    __graft_entry__.build()
    from long_context_anchor_gb300 import kascade
    return kascade


def _sim(L, seed):
    rng = np.random.default_rng(seed)
    X = rng.random((L, L))
    M = (X + X.T) / 2
    np.fill_diagonal(M, 1.0)
    return M


def test_round_trip_and_dp_objective(K, tmp_path):
    M = _sim(12, 3)
    anchors, f = K.schedule_anchors(M.tolist(), 4)
    path = str(tmp_path / "sched.json")
    doc = SF.save_schedule(path, anchors, M, meta={"topk": 4096, "calibration": "4 x 32768"})
    assert abs(doc["objective"] - f) < 1e-9
    back = SF.load_schedule(path)
    assert back["anchors"] == anchors and back["n_layers"] == 12
    assert np.array_equal(np.array(back["sim"]), M)
    assert abs(back["objective"] - f) < 1e-9
    assert back["meta"]["topk"] == 4096 and back["similarity"] == "overlap"


def test_objective_by_hand():
    # 4 layers, anchors {0, 2}: F = M[0][0] + M[0][1] + M[2][2] + M[2][3]
    M = [[1.0, 0.5, 0.1, 0.2], [0.5, 1.0, 0.3, 0.4], [0.1, 0.3, 1.0, 0.7], [0.2, 0.4, 0.7, 1.0]]
    assert SF.objective([0, 2], M) == pytest.approx(1.0 + 0.5 + 1.0 + 0.7)
    # a first anchor after layer 0: the dense layers before it add nothing
    assert SF.objective([1], M) == pytest.approx(1.0 + 0.3 + 0.4)


@pytest.mark.parametrize("anchors", [[], [0, 0], [2, 1], [0, 12], [-1], [0, 1.5], [True]])
def test_bad_anchor_lists_refused(tmp_path, anchors):
    with pytest.raises(SF.ScheduleError):
        SF.save_schedule(str(tmp_path / "s.json"), anchors, _sim(12, 1))


def test_bad_files_refused(tmp_path):
    M = _sim(6, 2)
    path = str(tmp_path / "s.json")
    SF.save_schedule(path, [0, 3], M, similarity="recall")
    good = json.load(open(path))

    def write(doc):
        with open(path, "w") as f:
            json.dump(doc, f)

    for mutate in (lambda d: d.update(format="other"),
                   lambda d: d.update(n_layers=7),
                   lambda d: d.update(anchors=[3, 0]),
                   lambda d: d.update(similarity="cosine"),
                   lambda d: d.update(objective=d["objective"] + 0.5),
                   lambda d: d["sim"][2].pop(),
                   lambda d: d["sim"][1].__setitem__(1, float("nan"))):
        doc = json.loads(json.dumps(good))
        mutate(doc)
        write(doc)
        with pytest.raises((SF.ScheduleError, ValueError)):
            SF.load_schedule(path)
    write(good)
    assert SF.load_schedule(path)["anchors"] == [0, 3]
    with pytest.raises(SF.ScheduleError):
        SF.save_schedule(path, [0], M, similarity="cosine")
