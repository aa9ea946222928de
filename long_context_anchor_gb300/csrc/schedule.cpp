// schedule.cpp — host dynamic programme that picks the anchor layers
// (Kascade, opentrain.ai Abstract: anchors are "selected algorithmically, via
// a dynamic-programming objective that maximizes cross-layer similarity";
// euno.news summary, Methodology 4).
//
// Objective: F(A) = sum over layers l of sim[a(l)][l], a(l) the most recent
// anchor at or before l, |A| = m, layer 0 always an anchor. With
// run(i, j) = sum_{l=i}^{j-1} sim[i][l] (anchor i serving layers i..j-1):
//   V[c][i] = best value of layers i..L-1 with an anchor at i and c anchors
//             in i..L-1;  V[1][i] = run(i, L);
//   V[c][i] = max_{j=i+1}^{L-c+1} run(i, j) + V[c-1][j].
// The list is rebuilt from layer 0, each time taking the smallest next
// anchor that keeps the optimum (ties -> lexicographically smallest list).
#include <math.h>
#include <stdint.h>

#include <vector>

#include "kascade.h"

extern "C" kascade_status kascade_schedule_anchors(const double* sim, int32_t n_layers,
                                                   int32_t n_anchors, int32_t* anchors_out,
                                                   double* objective_out) {
  if (sim == nullptr || anchors_out == nullptr) return KASCADE_ERR_INVALID_ARG;
  const int L = n_layers, m = n_anchors;
  if (L < 1 || m < 1 || m > L) return KASCADE_ERR_INVALID_ARG;
  for (int i = 0; i < L * L; ++i)
    if (!isfinite(sim[i])) return KASCADE_ERR_INVALID_ARG;
  // prefix sums along each anchor row: run(i, j) = P[i][j] - P[i][i]
  std::vector<double> P(static_cast<size_t>(L) * (L + 1), 0.0);
  for (int i = 0; i < L; ++i)
    for (int l = 0; l < L; ++l) P[i * (L + 1) + l + 1] = P[i * (L + 1) + l] + sim[i * L + l];
  auto run = [&](int i, int j) { return P[i * (L + 1) + j] - P[i * (L + 1) + i]; };
  const double kNone = -INFINITY;
  std::vector<double> V(static_cast<size_t>(m + 1) * L, kNone);
  for (int i = 0; i < L; ++i) V[1 * L + i] = run(i, L);
  for (int c = 2; c <= m; ++c) {
    for (int i = 0; i + c <= L; ++i) {
      double best = kNone;
      for (int j = i + 1; j <= L - c + 1; ++j) {
        const double cand = run(i, j) + V[(c - 1) * L + j];
        if (cand > best) best = cand;
      }
      V[c * L + i] = best;
    }
  }
  anchors_out[0] = 0;
  int cur = 0;
  for (int c = m, n = 1; c >= 2; --c, ++n) {
    const double target = V[c * L + cur];
    const double tol = 1e-12 * (fabs(target) > 1.0 ? fabs(target) : 1.0);
    int pick = -1;
    for (int j = cur + 1; j <= L - c + 1; ++j) {
      if (run(cur, j) + V[(c - 1) * L + j] >= target - tol) {
        pick = j;
        break;
      }
    }
    if (pick < 0) return KASCADE_ERR_INVALID_ARG;   // not reachable for finite input
    anchors_out[n] = pick;
    cur = pick;
  }
  if (objective_out) *objective_out = V[m * L + 0];
  return KASCADE_OK;
}
