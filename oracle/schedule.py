"""Cross-layer Top-k overlap and the anchor-selection dynamic programme (oracle).

The pages say the anchor layers are chosen "algorithmically, via a
dynamic-programming objective that maximizes cross-layer similarity over a
development set" (opentrain.ai, Abstract) and that the DP "maximizes the
overlap (similarity) of top-k sets across layers" (euno.news summary,
Methodology 4). Readings where they are silent:

* similarity of layer i to layer l: M[i][l] = mean over calibration
  (sequence, query head) of |S_i ∩ S_l| / k, where S_x is layer x's own exact
  Top-k (every layer run as an anchor on the calibration data);
* a reuse layer l follows the most recent anchor a(l) = max{a in A : a <= l};
* objective: F(A) = sum over layers l of M[a(l)][l], |A| = m, 0 in A
  (so M[l][l] = 1 counts each anchor fully);
* ties go to the lexicographically smallest anchor list.
"""
import numpy as np


def overlap_similarity(sets, k: int) -> np.ndarray:
    """sets[l][u] = index set of layer l for unit u (a (sequence, head) pair).

    Returns M [L, L] with M[i][l] = mean_u |S_i(u) ∩ S_l(u)| / k (symmetric).
    """
    L = len(sets)
    U = len(sets[0])
    M = np.zeros((L, L))
    as_sets = [[set(np.asarray(sets[l][u]).tolist()) for u in range(U)] for l in range(L)]
    for i in range(L):
        for l in range(i, L):
            tot = 0
            for u in range(U):
                tot += len(as_sets[i][u] & as_sets[l][u])
            M[i, l] = M[l, i] = tot / (U * k)
    return M


def objective(M, anchors) -> float:
    """F(A) = sum_l M[a(l)][l], a(l) the most recent anchor at or before l."""
    M = np.asarray(M, dtype=np.float64)
    L = M.shape[0]
    A = sorted(anchors)
    total = 0.0
    cur = None
    pos = 0
    for layer in range(L):
        while pos < len(A) and A[pos] <= layer:
            cur = A[pos]
            pos += 1
        if cur is None:
            raise ValueError("layer before the first anchor")
        total += M[cur, layer]
    return total


def schedule_anchors(M, m: int, rel_tol: float = 1e-12):
    """Anchor list of size m (containing 0) maximising ``objective``; ties lexicographic.

    Suffix recurrence: best[c][i] = best value of layers [i, L) given an anchor
    at i and c anchors in [i, L):
      best[1][i] = seg(i, L),
      best[c][i] = max_{i < j <= L-c+1} seg(i, j) + best[c-1][j],
    with seg(i, j) = sum_{l=i}^{j-1} M[i][l]. The list is rebuilt from 0 by
    taking, at each step, the smallest next anchor that keeps the optimum.
    """
    M = np.asarray(M, dtype=np.float64)
    L = M.shape[0]
    if not 1 <= m <= L:
        raise ValueError("need 1 <= m <= L")
    seg = np.zeros((L, L + 1))
    for i in range(L):
        acc = 0.0
        for j in range(i + 1, L + 1):
            acc += M[i, j - 1]
            seg[i, j] = acc
    NEG = -np.inf
    best = np.full((m + 1, L + 1), NEG)
    for i in range(L):
        best[1][i] = seg[i, L]
    for c in range(2, m + 1):
        for i in range(L):
            v = NEG
            for j in range(i + 1, L - c + 2):
                if best[c - 1][j] == NEG:
                    continue
                v = max(v, seg[i, j] + best[c - 1][j])
            best[c][i] = v
    anchors = [0]
    cur = 0
    for c in range(m, 1, -1):
        target = best[c][cur]
        tol = rel_tol * max(1.0, abs(target))
        for j in range(cur + 1, L - c + 2):
            if best[c - 1][j] != NEG and seg[cur, j] + best[c - 1][j] >= target - tol:
                anchors.append(j)
                cur = j
                break
    return anchors, float(best[m][0])


def mass_recall_similarity(probs, sets) -> np.ndarray:
    """Attention-mass recall between layers (an alternative DP similarity).

    The pages call the DP's quantity the "overlap (similarity) of top-k sets"
    without a formula (euno.news summary, Methodology 4). This variant asks how
    much of layer l's exact attention a set saved at layer i would keep:

        M[i][l] = mean over units u of sum_{j in S_i(u)} p_l(u)[j]

    with p_l(u) layer l's softmax weights over all keys for unit u (a
    (sequence, query head) pair) and S_i(u) the set layer i would hand to it.
    Entries lie in [0, 1]; M[l][l] is the mass a layer's own Top-k keeps. The
    DP reads M[i][l] only for i <= l. If p_l were uniform on S_l, M[i][l]
    would be |S_i ∩ S_l| / k, the overlap similarity.

    probs[l][u]: 1-D weights of layer l, unit u; sets[i][u]: index set.
    """
    L = len(probs)
    U = len(probs[0])
    M = np.zeros((L, L))
    for i in range(L):
        for l in range(L):
            tot = 0.0
            for u in range(U):
                sel = np.asarray(sets[i][u], dtype=np.int64)
                tot += float(np.asarray(probs[l][u], dtype=np.float64)[sel].sum())
            M[i, l] = tot / U
    return M
