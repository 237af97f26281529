// Rows of one batch shared out over several GPUs.
//
// A row is a tree of prompts, and a query sees only its own prompt
// (basal-rs Architecture page, "01 / Request path: Batch and prefix tree";
// "03 / Packing: Attention over tree blocks"), so the rows of a batch can be
// planned and run on different GPUs with no data exchanged between them.  Each
// GPU keeps a copy of the resident blocks (the template computed once at
// startup, "03 / Packing: Shared state computed once"), and the decisions are
// gathered on the host afterwards.
//
// Units of the split.  A row is the subtree of a non-resident block whose
// parent is resident or absent, after identical siblings have been merged (so
// rows that merge into one stay one).  Rows joined by a question (its two
// option-order leaves in different rows) form one unit, because the readout
// needs both.  A unit's cost is its visible (query, key) pairs per head: a
// query at position p sees p + 1 keys.  Units go to ranks longest-processing-
// time first: in decreasing cost (ties: the unit whose first row comes first in
// packed order), each to the rank with the least cost so far (ties: lowest rank).

#include <algorithm>
#include <cstring>
#include <numeric>
#include <vector>

#include "internal.h"

namespace {

int find(std::vector<int32_t> &up, int32_t x) {
  while (up[x] != x) {
    up[x] = up[up[x]];
    x = up[x];
  }
  return x;
}

}  // namespace

extern "C" {

int tree_shard_rows(const tree_spec_t *spec, const tree_plan_opts_t *opts, int32_t n_ranks, int32_t *block_rank,
                    int32_t *question_rank, int64_t *rank_pairs) {
  if (!spec || !block_rank || (spec->n_questions > 0 && !question_rank))
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_shard_rows: NULL argument");
  if (n_ranks <= 0) return tree::fail(TREE_ERR_INVALID_ARG, "tree_shard_rows: n_ranks %d", n_ranks);
  tree_plan_opts_t o{};
  if (opts) o = *opts;
  o.tiling = 0;  // the merged structure does not depend on the key tiling
  tree_plan_t *plan = nullptr;
  int rc = tree_pack_plan(spec, &o, &plan);
  if (rc != TREE_OK) return rc;
  const tree::Plan &P = plan->p;
  const int32_t nb = P.n_blocks;
  // row of every packed block (parents precede children in packed order)
  std::vector<int32_t> row(nb, -1);
  std::vector<int64_t> cost(nb, 0);
  for (int32_t b = 0; b < nb; ++b) {
    if (P.blk_resident[b]) continue;
    const int32_t par = P.blk_parent[b];
    row[b] = (par < 0 || P.blk_resident[par]) ? b : row[par];
    const int64_t L = P.blk_len[b], p0 = P.blk_pos0[b];
    cost[row[b]] += L * p0 + L * (L + 1) / 2;
  }
  // rows joined by a question are one unit
  std::vector<int32_t> up(nb);
  std::iota(up.begin(), up.end(), 0);
  for (int32_t q = 0; q < spec->n_questions; ++q) {
    const int32_t a = row[P.block_map[spec->leaf1[q]]], c = row[P.block_map[spec->leaf2[q]]];
    if (a < 0 || c < 0) {
      tree_plan_free(plan);
      return tree::fail(TREE_ERR_INVALID_ARG, "tree_shard_rows: question %d reads out a resident block", q);
    }
    const int32_t ra = find(up, a), rc2 = find(up, c);
    if (ra != rc2) up[std::max(ra, rc2)] = std::min(ra, rc2);  // the unit is named by its first row
  }
  std::vector<int64_t> unit_cost(nb, 0);
  std::vector<int32_t> units;
  for (int32_t b = 0; b < nb; ++b) {
    if (row[b] != b) continue;  // b heads a row
    const int32_t u = find(up, b);
    if (u == b) units.push_back(u);  // a unit's first row is the row it is named by
    unit_cost[u] += cost[b];
  }
  std::stable_sort(units.begin(), units.end(), [&](int32_t x, int32_t y) { return unit_cost[x] > unit_cost[y]; });
  std::vector<int64_t> load(n_ranks, 0);
  std::vector<int32_t> unit_rank(nb, -1);
  for (int32_t u : units) {
    const int32_t r = (int32_t)(std::min_element(load.begin(), load.end()) - load.begin());
    unit_rank[u] = r;
    load[r] += unit_cost[u];
  }
  for (int32_t i = 0; i < P.n_input_blocks; ++i) {
    const int32_t b = P.block_map[i];
    block_rank[i] = row[b] < 0 ? -1 : unit_rank[find(up, row[b])];
  }
  for (int32_t q = 0; q < spec->n_questions; ++q) question_rank[q] = unit_rank[find(up, row[P.block_map[spec->leaf1[q]]])];
  if (rank_pairs) std::memcpy(rank_pairs, load.data(), sizeof(int64_t) * n_ranks);
  tree_plan_free(plan);
  return TREE_OK;
}

int tree_shard_select(const tree_spec_t *spec, const int32_t *block_rank, const int32_t *question_rank, int32_t rank,
                      tree_shard_t *out) {
  if (!spec || !block_rank || !out || !out->parent || !out->length || !out->block_index ||
      (spec->n_questions > 0 && (!question_rank || !out->leaf1 || !out->leaf2 || !out->question_index)))
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_shard_select: NULL argument");
  if (spec->n_blocks <= 0 || !spec->parent || !spec->length)
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_shard_select: empty forest");
  const int32_t nb = spec->n_blocks;
  std::vector<int32_t> local(nb, -1);
  int32_t n = 0;
  for (int32_t b = 0; b < nb; ++b)
    if (block_rank[b] == rank || block_rank[b] == -1) local[b] = n++;
  n = 0;
  for (int32_t b = 0; b < nb; ++b) {
    if (local[b] < 0) continue;
    const int32_t par = spec->parent[b];
    if (par >= nb || (par >= 0 && local[par] < 0))
      return tree::fail(TREE_ERR_INVALID_ARG, "tree_shard_select: block %d kept without its parent %d", b, par);
    out->parent[n] = par < 0 ? -1 : local[par];
    out->length[n] = spec->length[b];
    if (out->key) out->key[n] = spec->key ? spec->key[b] : 0;
    if (out->resident) out->resident[n] = spec->resident ? spec->resident[b] : 0;
    out->block_index[n] = b;
    ++n;
  }
  out->n_blocks = n;
  int32_t m = 0;
  for (int32_t q = 0; q < spec->n_questions; ++q) {
    if (question_rank[q] != rank) continue;
    const int32_t a = spec->leaf1[q], c = spec->leaf2[q];
    if (a < 0 || a >= nb || c < 0 || c >= nb || local[a] < 0 || local[c] < 0)
      return tree::fail(TREE_ERR_INVALID_ARG, "tree_shard_select: question %d's leaves are not on rank %d", q, rank);
    out->leaf1[m] = local[a];
    out->leaf2[m] = local[c];
    out->question_index[m] = q;
    ++m;
  }
  out->n_questions = m;
  return TREE_OK;
}

}  // extern "C"
