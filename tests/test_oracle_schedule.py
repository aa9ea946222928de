"""Pins for oracle/schedule.py: the DP against exhaustive enumeration of
every anchor set, special cases (m = 1, m = L), a hand case, and the overlap
similarity against set arithmetic done by hand."""
import itertools

import numpy as np
import pytest

from oracle.schedule import objective, overlap_similarity, schedule_anchors


def _random_similarity(rng, L):
    # symmetric, unit diagonal, entries in (0, 1): like Top-k overlap fractions
    X = rng.random((L, L))
    M = (X + X.T) / 2
    np.fill_diagonal(M, 1.0)
    return M


def _exhaustive(M, m):
    L = M.shape[0]
    best, best_set = -np.inf, None
    for rest in itertools.combinations(range(1, L), m - 1):
        A = (0,) + rest
        f = objective(M, A)
        if f > best + 1e-12:            # combinations come in lexicographic order
            best, best_set = f, list(A)
    return best_set, best


@pytest.mark.parametrize("L,m", [(6, 1), (6, 2), (7, 3), (8, 4), (9, 9), (10, 5)])
def test_dp_equals_exhaustive_small(L, m):
    rng = np.random.default_rng(L * 10 + m)
    for _ in range(5):
        M = _random_similarity(rng, L)
        A, f = schedule_anchors(M, m)
        Ae, fe = _exhaustive(M, m)
        assert A == Ae
        np.testing.assert_allclose(f, fe, atol=1e-10)
        np.testing.assert_allclose(objective(M, A), f, atol=1e-10)


@pytest.mark.parametrize("L,m", [(6, 2), (7, 3), (8, 4), (9, 3), (10, 4)])
def test_dp_ties_pick_the_lexicographically_smallest_set(L, m):
    """Entries in {0, 1/2, 1} sum exactly in float64, so many anchor sets tie
    for the optimum; the DP must return the first of them in lexicographic
    order, as exhaustive enumeration does."""
    rng = np.random.default_rng(100 + L * 10 + m)
    n_tied = 0
    for _ in range(20):
        M = rng.integers(0, 3, size=(L, L)) / 2.0
        np.fill_diagonal(M, 1.0)
        A, f = schedule_anchors(M, m)
        Ae, fe = _exhaustive(M, m)
        assert A == Ae and f == fe
        vals = [objective(M, (0,) + rest) for rest in itertools.combinations(range(1, L), m - 1)]
        n_tied += sum(v == fe for v in vals) > 1
    assert n_tied > 0   # the cases do exercise ties


def test_dp_equals_exhaustive_L32_m6():
    """All C(31, 5) = 169,911 anchor sets of a 32-layer stack, vectorised."""
    rng = np.random.default_rng(32)
    L, m = 32, 6
    M = _random_similarity(rng, L)
    A, f = schedule_anchors(M, m)
    combos = np.array(list(itertools.combinations(range(1, L), m - 1)), dtype=np.int64)
    sets = np.concatenate([np.zeros((len(combos), 1), np.int64), combos], axis=1)
    # a(l) for each set and layer: the largest anchor <= l
    layers = np.arange(L)
    pos = np.zeros((len(sets), L), dtype=np.int64)
    for c in range(m):
        pos = np.where(sets[:, c:c + 1] <= layers[None, :], sets[:, c:c + 1], pos)
    F = M[pos, layers[None, :]].sum(axis=1)
    best = F.max()
    first = int(np.flatnonzero(F >= best - 1e-12)[0])
    assert A == sets[first].tolist()
    np.testing.assert_allclose(f, best, atol=1e-10)


def test_special_cases():
    rng = np.random.default_rng(0)
    M = _random_similarity(rng, 12)
    A, f = schedule_anchors(M, 1)
    assert A == [0]
    np.testing.assert_allclose(f, M[0].sum(), atol=1e-12)
    A, f = schedule_anchors(M, 12)
    assert A == list(range(12))
    np.testing.assert_allclose(f, 12.0, atol=1e-12)


def test_hand_case_two_blocks():
    # layers 0-3 resemble each other, 4-7 resemble each other, across blocks 0.
    L = 8
    M = np.zeros((L, L))
    M[:4, :4] = 0.9
    M[4:, 4:] = 0.9
    np.fill_diagonal(M, 1.0)
    A, f = schedule_anchors(M, 2)
    assert A == [0, 4]
    np.testing.assert_allclose(f, 2 * (1 + 3 * 0.9), atol=1e-12)
    # all-equal similarity: every placement ties; the smallest list wins
    A, _ = schedule_anchors(np.ones((5, 5)), 3)
    assert A == [0, 1, 2]


def test_overlap_similarity_by_hand():
    k = 4
    sets = [
        [[0, 1, 2, 3], [4, 5, 6, 7]],      # layer 0, two units
        [[0, 1, 8, 9], [4, 5, 6, 7]],      # layer 1
        [[10, 11, 12, 13], [7, 20, 21, 22]],  # layer 2
    ]
    M = overlap_similarity(sets, k)
    np.testing.assert_allclose(np.diag(M), 1.0)
    np.testing.assert_allclose(M[0, 1], (2 + 4) / 8)
    np.testing.assert_allclose(M[0, 2], (0 + 1) / 8)
    np.testing.assert_allclose(M[1, 2], (0 + 1) / 8)
    assert (M == M.T).all()


# ------------------------------------------------- mass-recall similarity --

from oracle.schedule import mass_recall_similarity  # noqa: E402
from oracle.topk import topk_indices  # noqa: E402


def _softmax_rows(rng, L, U, N, scale=2.0):
    x = scale * rng.standard_normal((L, U, N))
    e = np.exp(x - x.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


def test_mass_recall_diagonal_is_topk_mass_and_bounds():
    rng = np.random.default_rng(31)
    L, U, N, k = 4, 5, 60, 7
    p = _softmax_rows(rng, L, U, N)
    sets = [[topk_indices(p[l, u], k) for u in range(U)] for l in range(L)]
    M = mass_recall_similarity(p, sets)
    for l in range(L):
        # the k largest weights of each unit, summed and averaged
        top = np.sort(p[l], axis=-1)[:, ::-1][:, :k].sum(-1).mean()
        np.testing.assert_allclose(M[l, l], top, atol=1e-14)
        # no other set of k keys keeps more of layer l's mass
        assert (M[:, l] <= M[l, l] + 1e-14).all()
    assert (M >= 0).all() and (M <= 1 + 1e-12).all()


def test_mass_recall_full_sets_and_uniform_weights_give_overlap():
    rng = np.random.default_rng(32)
    L, U, N, k = 3, 4, 40, 9
    # k = N keeps all mass
    p = _softmax_rows(rng, L, U, N)
    full = [[np.arange(N) for _ in range(U)] for _ in range(L)]
    np.testing.assert_allclose(mass_recall_similarity(p, full), 1.0, atol=1e-12)
    # weights uniform on the layer's own set: recall is the overlap fraction
    sets = [[np.sort(rng.choice(N, k, replace=False)) for _ in range(U)] for _ in range(L)]
    pu = np.zeros((L, U, N))
    for l in range(L):
        for u in range(U):
            pu[l, u, sets[l][u]] = 1.0 / k
    np.testing.assert_allclose(mass_recall_similarity(pu, sets), overlap_similarity(sets, k),
                               atol=1e-12)


def test_mass_recall_drives_the_dp():
    # layers 0-2 attend to one key group, 3-5 to another: the recall matrix
    # is block-structured and two anchors go to 0 and 3
    N, U, k = 32, 3, 4
    p = np.full((6, U, N), 1e-4)
    for l in range(6):
        keys = [0, 1, 2, 3] if l < 3 else [16, 17, 18, 19]
        p[l][:, keys] = 1.0
    p /= p.sum(-1, keepdims=True)
    sets = [[topk_indices(p[l, u], k) for u in range(U)] for l in range(6)]
    M = mass_recall_similarity(p, sets)
    A, _ = schedule_anchors(M, 2)
    assert A == [0, 3]
