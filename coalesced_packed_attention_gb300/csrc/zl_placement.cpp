// Host placement slice of the two-stage planner (no GPU): the catalog cut that
// separates anchor buckets from filler buckets, and the greedy packing of whole filler
// sequences into the per-rank headroom left by the anchors ("Zellige", pith.science
// review, "Free parameters" and the referee report on Eq. (8): the cut is the Fisher
// grouping under which the log run times of whole sequences vary least inside each
// set; a filler goes to the rank whose tighter resource, compute headroom against F or
// memory headroom against M_cap, stays the most open).
//
// Catalog cut.  Buckets sorted by whole-sequence time T_1 <= ... <= T_B, bucket b
// holding n_b sequences.  For a cut k in 1..B-1 the fillers are buckets 1..k and the
// anchors k+1..B; with x_b = ln T_b,
//   D(k) = sum_{b<=k} n_b (x_b - mu_F)^2 + sum_{b>k} n_b (x_b - mu_A)^2,
// mu_F, mu_A the count-weighted means of x over each side.  k* = argmin D (smallest k
// on ties).  One bucket: k* = 1, every sequence a filler, D = 0.
//
// Filler packing.  Fillers in decreasing time (ties: lower index first).  Each goes to
// the rank with the largest bottleneck score
//   score_r = min((F - L_r - t) / F, (M_cap - M_r - m) / M_cap)
// (ties: lowest rank), where L_r, M_r are the rank's time and memory so far (anchors
// first).  A filler whose best score is below -1e-9 (negative beyond the rounding of an
// exact fit) still goes there and is counted as an overflow.  F <= 0 selects the
// makespan lower bound max(max_r L_r, sum of all time / N).
#include <algorithm>
#include <cmath>
#include <numeric>
#include <vector>

#include "zl_internal.h"

namespace {

bool finite_pos(double x) { return std::isfinite(x) && x > 0.0; }

}  // namespace

extern "C" zl_status zl_catalog_cut(const zl_bucket* buckets, int32_t n_buckets, int32_t* k_star,
                                    double* dispersion) {
  if (!buckets || n_buckets < 1 || !k_star) return ZL_ERR_INVALID_ARG;
  for (int32_t b = 0; b < n_buckets; ++b) {
    if (buckets[b].count < 1 || !finite_pos(buckets[b].time)) return ZL_ERR_INVALID_ARG;
    if (b > 0 && buckets[b].time < buckets[b - 1].time) return ZL_ERR_INVALID_ARG;  // must be sorted
  }
  if (n_buckets == 1) {
    *k_star = 1;
    if (dispersion) *dispersion = 0.0;
    return ZL_OK;
  }
  // prefix sums of n, n x, n x^2 (x = ln T); each side's sum of squared deviations is
  // S2 - S1^2 / S0
  std::vector<double> s0(n_buckets + 1, 0.0), s1(n_buckets + 1, 0.0), s2(n_buckets + 1, 0.0);
  for (int32_t b = 0; b < n_buckets; ++b) {
    const double n = buckets[b].count, x = std::log(buckets[b].time);
    s0[b + 1] = s0[b] + n;
    s1[b + 1] = s1[b] + n * x;
    s2[b + 1] = s2[b] + n * x * x;
  }
  auto ssd = [&](int32_t lo, int32_t hi) {  // buckets [lo, hi)
    const double n = s0[hi] - s0[lo], a = s1[hi] - s1[lo], q = s2[hi] - s2[lo];
    const double v = q - a * a / n;
    return v > 0.0 ? v : 0.0;
  };
  int32_t best = 1;
  double best_d = ssd(0, 1) + ssd(1, n_buckets);
  for (int32_t k = 2; k < n_buckets; ++k) {
    const double d = ssd(0, k) + ssd(k, n_buckets);
    if (d < best_d) {
      best_d = d;
      best = k;
    }
  }
  *k_star = best;
  if (dispersion) *dispersion = best_d;
  return ZL_OK;
}

extern "C" zl_status zl_pack_fillers(const double* filler_time, const double* filler_mem, int32_t n_fillers,
                                     int32_t n_ranks, const double* rank_time, const double* rank_mem, double F,
                                     double M_cap, int32_t* assign, double* final_time, double* final_mem,
                                     int32_t* n_overflow, double* makespan) {
  if (n_fillers < 0 || n_ranks < 1 || (n_fillers > 0 && (!filler_time || !filler_mem || !assign)))
    return ZL_ERR_INVALID_ARG;
  if (!finite_pos(M_cap) || !std::isfinite(F)) return ZL_ERR_INVALID_ARG;
  std::vector<double> L(n_ranks, 0.0), M(n_ranks, 0.0);
  for (int32_t r = 0; r < n_ranks; ++r) {
    if (rank_time) L[r] = rank_time[r];
    if (rank_mem) M[r] = rank_mem[r];
    if (!std::isfinite(L[r]) || !std::isfinite(M[r]) || L[r] < 0.0 || M[r] < 0.0) return ZL_ERR_INVALID_ARG;
  }
  double total = std::accumulate(L.begin(), L.end(), 0.0);
  for (int32_t s = 0; s < n_fillers; ++s) {
    if (!std::isfinite(filler_time[s]) || filler_time[s] < 0.0 || !std::isfinite(filler_mem[s]) ||
        filler_mem[s] < 0.0)
      return ZL_ERR_INVALID_ARG;
    total += filler_time[s];
  }
  if (F <= 0.0) F = std::max(*std::max_element(L.begin(), L.end()), total / n_ranks);
  if (!finite_pos(F)) F = 1.0;  // nothing to place and nothing placed: any positive scale
  std::vector<int32_t> order(n_fillers);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return filler_time[a] > filler_time[b]; });
  int32_t over = 0;
  for (int32_t s : order) {
    const double t = filler_time[s], m = filler_mem[s];
    int32_t best = 0;
    double best_score = -INFINITY;
    for (int32_t r = 0; r < n_ranks; ++r) {
      const double score = std::min((F - L[r] - t) / F, (M_cap - M[r] - m) / M_cap);
      if (score > best_score) {
        best_score = score;
        best = r;
      }
    }
    if (best_score < -1e-9) ++over;
    assign[s] = best;
    L[best] += t;
    M[best] += m;
  }
  if (final_time) std::copy(L.begin(), L.end(), final_time);
  if (final_mem) std::copy(M.begin(), M.end(), final_mem);
  if (n_overflow) *n_overflow = over;
  if (makespan) *makespan = *std::max_element(L.begin(), L.end());
  return ZL_OK;
}
