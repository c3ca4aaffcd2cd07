// Host-side partition of a matrix set across data-parallel ranks (declared in include/muon.h).
//
// The speedrun reduce-scatters gradients instead of all-reducing them (energy-efficiency article on
// Modded-NanoGPT, technical-evolution section; "How to train a GPT model in 3 minutes", section on
// system optimisations, distributed communication), and puts the attention and MLP parameters
// into one reduce_scatter call (the "Muon Custom Sizing" article in the related-article list of
// the record analysis of 2026-05-27_MuddGatedAndDC). Every matrix's Newton-Schulz iteration is
// independent, so the unit of work here is a whole matrix: each rank owns a subset, receives the
// summed gradient of exactly that subset from one reduce-scatter over all matrices, runs muon_step
// on it, and one all-gather returns every rank's updated parameters to all ranks (replicated
// parameters, as the record analysis' optimizer table calls the communication mode of the
// parameters every rank keeps whole).
//
// This file only decides who owns what and where each matrix sits in the flat rank-major buffers
// the two collectives work on in place. No GPU is touched.
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "../../include/muon.h"

namespace {

// Algorithmic flops of one Newton-Schulz iteration on a rows x cols matrix: n(n+1)m for the
// upper-triangle Gram, 2 n^2 m for B X, and n^2(n+1) for A A when c != 0 (n = min, m = max).
double iteration_flops(int64_t rows, int64_t cols, bool with_c) {
  if (rows <= 0 || cols <= 0) return 0.0;
  const double n = static_cast<double>(std::min(rows, cols)), m = static_cast<double>(std::max(rows, cols));
  return n * (n + 1.0) * m + 2.0 * n * n * m + (with_c ? n * n * (n + 1.0) : 0.0);
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

extern "C" muon_status muon_shard_layout(const int64_t* rows, const int64_t* cols, int count, int world, int with_c,
                                         int64_t align, int* owner, int64_t* offset, int64_t* segment,
                                         double* load) {
  if (count < 0 || world < 1 || align < 1 || (count > 0 && (!rows || !cols || !owner || !offset)) || !segment)
    return MUON_ERR_INVALID;
  for (int j = 0; j < count; ++j)
    if (rows[j] < 0 || cols[j] < 0) return MUON_ERR_INVALID;

  // Longest processing time first: matrices by decreasing flops (index breaks ties), each to the
  // rank with the least flops so far (lowest rank breaks ties). Empty matrices cost nothing and go
  // to rank 0.
  std::vector<int> order(static_cast<size_t>(count));
  std::iota(order.begin(), order.end(), 0);
  std::vector<double> cost(static_cast<size_t>(count));
  for (int j = 0; j < count; ++j) cost[j] = iteration_flops(rows[j], cols[j], with_c != 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });
  std::vector<double> sum(static_cast<size_t>(world), 0.0);
  for (int j : order) {
    int best = 0;
    for (int r = 1; r < world; ++r)
      if (sum[r] < sum[best]) best = r;
    owner[j] = best;
    sum[best] += cost[j];
  }

  // Rank r's matrices sit in index order in its segment [r * segment, (r + 1) * segment) of the
  // flat buffers; every matrix starts on a multiple of `align` elements and every segment has the
  // same length, as an in-place reduce-scatter and all-gather require.
  std::vector<int64_t> fill(static_cast<size_t>(world), 0);
  for (int j = 0; j < count; ++j) {
    offset[j] = fill[owner[j]];
    fill[owner[j]] = round_up(fill[owner[j]] + rows[j] * cols[j], align);
  }
  int64_t seg = align;
  for (int r = 0; r < world; ++r) seg = std::max(seg, fill[r]);
  seg = round_up(seg, align);
  for (int j = 0; j < count; ++j) offset[j] += static_cast<int64_t>(owner[j]) * seg;
  *segment = seg;
  if (load)
    for (int r = 0; r < world; ++r) load[r] = sum[r];
  return MUON_OK;
}
