// Batch-aware draft budget: choose the tree's k and m for a batch size from measured costs.
//
// The pages observe that speedups shrink at large batch sizes, where verifying big trees costs
// real compute ("EAGLE: Feature-Level Drafting", paragraph "Common mistakes and limits"), and
// that a fixed k and m can mismatch the active batch or device ("EAGLE-2" page, table "Where
// It Breaks", row "Fixed k and m mismatch runtime capacity"). The drafter is calibrated, so a
// node's path value V estimates the chance that verification keeps it ("EAGLE-2" page, "Path
// Value Ranks Prefixes"): a tree of the m best nodes is expected to commit 1 + (sum of their
// V) tokens.
// A cycle of batch B costs the draft (depending on k) plus a verify pass over B (m + 1)
// rows, which is flat while the weight stream bounds it and grows once arithmetic does.
// The plan maximises B * E[tokens](k, m) / (draft(k) + verify(B (m + 1))).
//
// Host-only arithmetic over caller-supplied measurements; no device work.
#include <cmath>
#include <cstdint>

#include "eagle.h"
#include "eagle_ops.h"

namespace {

// Piecewise-linear interpolation of the measured verify time at `rows` (extrapolated
// linearly past the last point from the last two, held flat before the first).
double verify_at(int n_points, const int32_t* rows_pts, const float* us_pts, double rows) {
  // one point: flat up to it, proportional to the rows past it
  if (n_points == 1) return us_pts[0] * std::fmax(1.0, rows / rows_pts[0]);
  if (rows <= rows_pts[0]) return us_pts[0];
  for (int i = 1; i < n_points; ++i) {
    if (rows <= rows_pts[i]) {
      const double f = (rows - rows_pts[i - 1]) / (double)(rows_pts[i] - rows_pts[i - 1]);
      return us_pts[i - 1] + f * (us_pts[i] - us_pts[i - 1]);
    }
  }
  const int a = n_points - 2, b = n_points - 1;
  const double slope = (us_pts[b] - us_pts[a]) / (double)(rows_pts[b] - rows_pts[a]);
  return us_pts[b] + std::fmax(0.0, slope) * (rows - rows_pts[b]);
}

}  // namespace

extern "C" int eagle_plan_budget(int n_k, const int32_t* k_values, const float* draft_us, const int32_t* m_max,
                                 const float* exp_tokens, int n_points, const int32_t* rows_pts,
                                 const float* verify_us, int batch, int32_t* best_k, int32_t* best_m,
                                 float* tokens_per_us) {
  if (n_k < 1 || !k_values || !draft_us || !m_max || !exp_tokens || n_points < 1 || !rows_pts || !verify_us ||
      batch < 1 || !best_k || !best_m)
    return EAGLE_EINVAL;
  for (int i = 0; i < n_points; ++i)
    if (rows_pts[i] < 1 || verify_us[i] <= 0.f || (i > 0 && rows_pts[i] <= rows_pts[i - 1])) return EAGLE_EINVAL;
  double best = -1.0;
  int bk = -1, bm = -1;
  size_t off = 0;
  for (int j = 0; j < n_k; ++j) {
    if (m_max[j] < 1 || draft_us[j] < 0.f) return EAGLE_EINVAL;
    for (int m = 1; m <= m_max[j]; ++m) {
      const double tok = exp_tokens[off + m - 1];
      const double t = draft_us[j] + verify_at(n_points, rows_pts, verify_us, (double)batch * (m + 1));
      const double rate = batch * tok / t;
      if (rate > best) {   // ties keep the smaller budget (listed k first, then smaller m)
        best = rate;
        bk = k_values[j];
        bm = m;
      }
    }
    off += (size_t)m_max[j];
  }
  *best_k = bk;
  *best_m = bm;
  if (tokens_per_us) *tokens_per_us = (float)best;
  return EAGLE_OK;
}
