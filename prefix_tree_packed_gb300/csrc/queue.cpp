// Host request planner: HRRN / FIFO queue with a long-request lane, batches
// packed as prefix-tree forests (basal-rs Architecture page, "01 / Request
// path": Validation and planning, HRRN queue, Batch and prefix tree; "04 /
// Scheduling").
//
// A request's prompts are root-to-leaf paths of blocks.  Its cost is the token
// count of the trie of its prompts (blocks with equal non-zero key and length
// under the same parent are one node; resident roots are free).  The next
// batch starts with the queued short request of highest priority and takes
// every further short request, in priority order, that fits: the trie of the
// whole batch (shared prefixes counted once across requests) stays within
// max_batch_tokens and every row (root) within max_row.

#include <algorithm>
#include <cstring>
#include <map>
#include <tuple>
#include <unordered_set>

#include "internal.h"
#include "tree_queue.h"

namespace tree {
namespace {

struct Request {
  int64_t id = 0;
  double arrival = 0.0;
  uint64_t seq = 0;  // push order: the last tie-break
  std::vector<int32_t> prompt_blocks;
  std::vector<tree_block_t> blocks;
  std::vector<int32_t> q1, q2;
  int64_t cost = 0;
};

// Prefix trie over prompts.  Nodes are created in first-seen order, so a
// parent always precedes its children.  Row sizes (tokens per root, resident
// blocks included), rows above the limit and resident roots are kept up to
// date, and a trial addition can be undone: every change it makes is a node
// appended at the end, a child count of an earlier node, a map entry keyed by
// the new node's own (parent, key, length), or a row total.
struct Trie {
  std::vector<int32_t> parent, length, resident, n_children, root;
  std::vector<uint64_t> key;
  std::vector<int64_t> row;  // per node: tokens of the row it roots (roots only)
  std::map<std::tuple<int32_t, uint64_t, int32_t>, int32_t> child;  // (parent, key, length) -> node
  int64_t cost = 0;
  int64_t max_row = INT64_MAX;
  int32_t res_roots = 0, over_rows = 0;

  size_t size() const { return parent.size(); }

  // Walk/extend the path of one prompt; returns its last node.
  int32_t add(const tree_block_t *b, int32_t n, const std::unordered_set<uint64_t> &res_keys) {
    int32_t p = -1;
    for (int32_t i = 0; i < n; ++i) {
      const auto k = std::make_tuple(p, b[i].key, b[i].length);
      auto it = b[i].key != 0 ? child.find(k) : child.end();
      if (it != child.end()) {
        p = it->second;
        continue;
      }
      const int32_t node = (int32_t)parent.size();
      const bool res = p < 0 && b[i].key != 0 && res_keys.count(b[i].key) > 0;
      parent.push_back(p);
      length.push_back(b[i].length);
      key.push_back(b[i].key);
      resident.push_back(res ? 1 : 0);
      n_children.push_back(0);
      root.push_back(p < 0 ? node : root[(size_t)p]);
      row.push_back(0);
      if (p >= 0) ++n_children[(size_t)p];
      if (b[i].key != 0) child.emplace(k, node);
      if (!res) cost += b[i].length;
      if (p < 0 && res) ++res_roots;
      int64_t &rw = row[(size_t)root[(size_t)node]];
      if (rw <= max_row && rw + b[i].length > max_row) ++over_rows;
      rw += b[i].length;
      p = node;
    }
    return p;
  }

  // Back to the state with n0 nodes and the given cost.
  void undo(size_t n0, int64_t cost0) {
    for (size_t n = size(); n-- > n0;) {
      if (key[n] != 0) child.erase(std::make_tuple(parent[n], key[n], length[n]));
      if (parent[n] >= 0) --n_children[(size_t)parent[n]];
      int64_t &rw = row[(size_t)root[n]];
      if (rw > max_row && rw - length[n] <= max_row) --over_rows;
      rw -= length[n];
      if (parent[n] < 0 && resident[n]) --res_roots;
    }
    for (auto *v : {&parent, &length, &resident, &n_children, &root}) v->resize(n0);
    key.resize(n0);
    row.resize(n0);
    cost = cost0;
  }
};

}  // namespace
}  // namespace tree

struct tree_queue {
  tree_queue_opts_t opts{};
  std::vector<uint64_t> resident_keys;
  std::unordered_set<uint64_t> res_set;
  std::vector<tree::Request> lane[2];  // 0 short, 1 long
  std::unordered_set<int64_t> ids;      // ids of the queued requests
  uint64_t next_seq = 0;
};

struct tree_batch {
  int32_t lane = 0;
  std::vector<int64_t> ids;
  std::vector<int32_t> q0;
  int64_t cost = 0;
  std::vector<int32_t> parent, length, leaf1, leaf2;
  std::vector<uint64_t> key;
  std::vector<uint8_t> resident;
};

namespace tree {
namespace {

// Adds every prompt of r to t; the readout node of each question prompt goes
// to leaves.  False if a readout node is (or becomes) an inner node, or if a
// row outgrows max_row, or a second resident root appears.
bool add_request(Trie &t, const Request &r, const tree_queue &q, std::vector<int32_t> &readout,
                 std::vector<int32_t> &leaf1, std::vector<int32_t> &leaf2) {
  t.max_row = q.opts.max_row;
  std::vector<int32_t> last(r.prompt_blocks.size());
  size_t off = 0;
  for (size_t p = 0; p < r.prompt_blocks.size(); ++p) {
    last[p] = t.add(r.blocks.data() + off, r.prompt_blocks[p], q.res_set);
    off += (size_t)r.prompt_blocks[p];
  }
  for (size_t i = 0; i < r.q1.size(); ++i) {
    leaf1.push_back(last[(size_t)r.q1[i]]);
    leaf2.push_back(last[(size_t)r.q2[i]]);
    readout.push_back(last[(size_t)r.q1[i]]);
    readout.push_back(last[(size_t)r.q2[i]]);
  }
  for (int32_t n : readout)
    if (t.n_children[(size_t)n] != 0) return false;
  return t.over_rows == 0 && t.res_roots <= 1;
}

// Schedule order of a lane at time now: highest priority first (HRRN) or
// earliest arrival (FIFO); ties by arrival, then push order.
std::vector<size_t> order_of(const std::vector<Request> &lane, const tree_queue &q, double now) {
  std::vector<size_t> idx(lane.size());
  for (size_t i = 0; i < idx.size(); ++i) idx[i] = i;
  auto prio = [&](const Request &r) {
    const double est = (double)std::max<int64_t>(r.cost, 1) * q.opts.ms_per_token;
    const double wait = std::max(0.0, now - r.arrival);
    return (wait + est) / est;
  };
  std::stable_sort(idx.begin(), idx.end(), [&](size_t a, size_t b) {
    const Request &ra = lane[a], &rb = lane[b];
    if (!q.opts.fifo) {
      const double pa = prio(ra), pb = prio(rb);
      if (pa != pb) return pa > pb;
    }
    if (ra.arrival != rb.arrival) return ra.arrival < rb.arrival;
    return ra.seq < rb.seq;
  });
  return idx;
}

}  // namespace
}  // namespace tree

using namespace tree;

extern "C" TREE_API int tree_queue_default_opts(tree_queue_opts_t *o) {
  if (!o) return fail(TREE_ERR_INVALID_ARG, "tree_queue_default_opts: NULL");
  std::memset(o, 0, sizeof(*o));
  o->max_batch_tokens = 8192;
  o->long_tokens = 4096;
  o->fifo = 0;
  o->ms_per_token = 0.01;
  o->max_depth = 8;
  o->max_row = 32768;
  return ok();
}

extern "C" TREE_API int tree_queue_create(const tree_queue_opts_t *o, tree_queue_t **out) {
  if (!o || !out) return fail(TREE_ERR_INVALID_ARG, "tree_queue_create: NULL argument");
  *out = nullptr;
  if (o->max_batch_tokens <= 0 || o->long_tokens < 0 || !(o->ms_per_token > 0.0) || o->max_depth <= 0 ||
      o->max_row <= 0 || o->n_resident < 0 || (o->n_resident > 0 && !o->resident_keys))
    return fail(TREE_ERR_INVALID_ARG, "tree_queue_create: bad options");
  auto *q = new tree_queue;
  q->opts = *o;
  q->resident_keys.assign(o->resident_keys, o->resident_keys + o->n_resident);
  q->opts.resident_keys = q->resident_keys.data();
  for (uint64_t k : q->resident_keys)
    if (k != 0) q->res_set.insert(k);
  *out = q;
  return ok();
}

extern "C" TREE_API int tree_queue_destroy(tree_queue_t *q) {
  delete q;
  return ok();
}

extern "C" TREE_API int tree_queue_push(tree_queue_t *q, const tree_request_t *r, int64_t *cost_out) {
  if (!q || !r) return fail(TREE_ERR_INVALID_ARG, "tree_queue_push: NULL argument");
  if (r->n_prompts < 1 || !r->prompt_blocks || !r->blocks || r->n_questions < 0 ||
      (r->n_questions > 0 && (!r->q_prompt1 || !r->q_prompt2)))
    return fail(TREE_ERR_INVALID_ARG, "tree_queue_push: bad counts or NULL arrays");
  if (q->ids.count(r->id)) return fail(TREE_ERR_INVALID_ARG, "tree_queue_push: id %lld already queued", (long long)r->id);
  Request req;
  req.id = r->id;
  req.arrival = r->arrival_ms;
  req.prompt_blocks.assign(r->prompt_blocks, r->prompt_blocks + r->n_prompts);
  size_t nb = 0;
  for (int32_t p = 0; p < r->n_prompts; ++p) {
    const int32_t n = req.prompt_blocks[(size_t)p];
    if (n < 1) return fail(TREE_ERR_INVALID_ARG, "tree_queue_push: prompt %d has %d blocks", p, n);
    if (n > q->opts.max_depth) return fail(TREE_ERR_DEPTH, "tree_queue_push: prompt %d has %d blocks > %d", p, n, q->opts.max_depth);
    int64_t tokens = 0;
    for (int32_t i = 0; i < n; ++i) {
      const int32_t len = r->blocks[nb + (size_t)i].length;
      if (len <= 0) return fail(TREE_ERR_BAD_TREE, "tree_queue_push: prompt %d block %d has length %d", p, i, len);
      tokens += len;
    }
    if (tokens > q->opts.max_row)
      return fail(TREE_ERR_ROW_TOO_LONG, "tree_queue_push: prompt %d has %lld tokens > %d", p, (long long)tokens, q->opts.max_row);
    nb += (size_t)n;
  }
  req.blocks.assign(r->blocks, r->blocks + nb);
  for (int32_t i = 0; i < r->n_questions; ++i) {
    const int32_t a = r->q_prompt1[i], b = r->q_prompt2[i];
    if (a < 0 || a >= r->n_prompts || b < 0 || b >= r->n_prompts)
      return fail(TREE_ERR_INVALID_ARG, "tree_queue_push: question %d names prompts %d, %d of %d", i, a, b, r->n_prompts);
    req.q1.push_back(a);
    req.q2.push_back(b);
  }
  // cost and the request's own readout nodes
  Trie t;
  std::vector<int32_t> readout, l1, l2;
  if (!add_request(t, req, *q, readout, l1, l2)) {
    for (int32_t n : readout)
      if (t.n_children[(size_t)n] != 0)
        return fail(TREE_ERR_INVALID_ARG, "tree_queue_push: a question prompt is a strict prefix of another prompt");
    return fail(TREE_ERR_ROW_TOO_LONG, "tree_queue_push: a row of the request exceeds %d tokens or has two resident roots",
                q->opts.max_row);
  }
  req.cost = t.cost;
  req.seq = q->next_seq++;
  const int lane = (q->opts.long_tokens > 0 && req.cost > q->opts.long_tokens) ? 1 : 0;
  if (cost_out) *cost_out = req.cost;
  q->ids.insert(req.id);
  q->lane[lane].push_back(std::move(req));
  return ok();
}

extern "C" TREE_API int tree_queue_cancel(tree_queue_t *q, int64_t id) {
  if (!q) return fail(TREE_ERR_INVALID_ARG, "tree_queue_cancel: NULL queue");
  for (auto &lane : q->lane)
    for (size_t i = 0; i < lane.size(); ++i)
      if (lane[i].id == id) {
        lane.erase(lane.begin() + (std::ptrdiff_t)i);
        q->ids.erase(id);
        return ok();
      }
  return fail(TREE_ERR_INVALID_ARG, "tree_queue_cancel: id %lld is not queued", (long long)id);
}

extern "C" TREE_API int tree_queue_info(const tree_queue_t *q, tree_queue_info_t *info) {
  if (!q || !info) return fail(TREE_ERR_INVALID_ARG, "tree_queue_info: NULL argument");
  info->n_short = (int32_t)q->lane[0].size();
  info->n_long = (int32_t)q->lane[1].size();
  return ok();
}

extern "C" TREE_API int tree_queue_pop(tree_queue_t *q, double now_ms, tree_batch_t **out) {
  if (!q || !out) return fail(TREE_ERR_INVALID_ARG, "tree_queue_pop: NULL argument");
  *out = nullptr;
  const int lane = !q->lane[0].empty() ? 0 : (!q->lane[1].empty() ? 1 : -1);
  if (lane < 0) return ok();
  auto &reqs = q->lane[lane];
  const std::vector<size_t> order = order_of(reqs, *q, now_ms);
  Trie t;
  std::vector<int32_t> readout, leaf1, leaf2;
  std::vector<size_t> taken;
  std::vector<int32_t> q0{0};
  for (size_t k = 0; k < order.size(); ++k) {
    const Request &r = reqs[order[k]];
    if (k == 0) {
      add_request(t, r, *q, readout, leaf1, leaf2);  // the first request is always taken (checked at push)
    } else {
      if (lane == 1) break;  // a long request runs alone
      // try it in place; a request that does not fit is undone
      const size_t n0 = t.size(), r0 = readout.size(), l0 = leaf1.size();
      const int64_t c0 = t.cost;
      if (!add_request(t, r, *q, readout, leaf1, leaf2) || t.cost > q->opts.max_batch_tokens) {
        t.undo(n0, c0);
        readout.resize(r0);
        leaf1.resize(l0);
        leaf2.resize(l0);
        continue;
      }
    }
    taken.push_back(order[k]);
    q0.push_back((int32_t)leaf1.size());
  }
  auto *b = new tree_batch;
  b->lane = lane;
  b->cost = t.cost;
  for (size_t i : taken) {
    b->ids.push_back(reqs[i].id);
    q->ids.erase(reqs[i].id);
  }
  b->q0 = q0;
  // the resident root (at most one) goes first, so that its tokens lead the
  // packed row; every other block keeps its first-seen place (parents first)
  const size_t nn = t.parent.size();
  std::vector<int32_t> perm;  // new index -> old
  for (size_t n = 0; n < nn; ++n)
    if (t.parent[n] < 0 && t.resident[n]) perm.push_back((int32_t)n);
  for (size_t n = 0; n < nn; ++n)
    if (!(t.parent[n] < 0 && t.resident[n])) perm.push_back((int32_t)n);
  std::vector<int32_t> inv(nn);
  for (size_t i = 0; i < nn; ++i) inv[(size_t)perm[i]] = (int32_t)i;
  for (size_t i = 0; i < nn; ++i) {
    const size_t o = (size_t)perm[i];
    b->parent.push_back(t.parent[o] < 0 ? -1 : inv[(size_t)t.parent[o]]);
    b->length.push_back(t.length[o]);
    b->key.push_back(t.key[o]);
    b->resident.push_back((uint8_t)t.resident[o]);
  }
  for (int32_t x : leaf1) b->leaf1.push_back(inv[(size_t)x]);
  for (int32_t x : leaf2) b->leaf2.push_back(inv[(size_t)x]);
  std::sort(taken.begin(), taken.end());
  for (size_t k = taken.size(); k-- > 0;) reqs.erase(reqs.begin() + (std::ptrdiff_t)taken[k]);
  *out = b;
  return ok();
}

extern "C" TREE_API int tree_batch_view(const tree_batch_t *b, tree_batch_view_t *v) {
  if (!b || !v) return fail(TREE_ERR_INVALID_ARG, "tree_batch_view: NULL argument");
  std::memset(v, 0, sizeof(*v));
  v->lane = b->lane;
  v->n_requests = (int32_t)b->ids.size();
  v->request_ids = b->ids.data();
  v->request_q0 = b->q0.data();
  v->cost = b->cost;
  v->spec.n_blocks = (int32_t)b->parent.size();
  v->spec.parent = b->parent.data();
  v->spec.length = b->length.data();
  v->spec.key = b->key.data();
  v->spec.resident = b->resident.data();
  v->spec.n_questions = (int32_t)b->leaf1.size();
  v->spec.leaf1 = b->leaf1.data();
  v->spec.leaf2 = b->leaf2.data();
  return ok();
}

extern "C" TREE_API int tree_batch_free(tree_batch_t *b) {
  delete b;
  return ok();
}
