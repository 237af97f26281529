// Host planner: a batch's prompt blocks -> prefix trees -> one packed token row.
//
// Follows the basal-rs Architecture page: "01 / Request path: Batch and prefix
// tree" (rows are trees whose shared prefixes are computed once; at most
// 32,768 tokens per row, 8192 per forward, 8 blocks deep; identical prompts
// share one readout) and "03 / Packing: Attention over tree blocks" (the tree
// becomes one row of tokens; a token sees earlier tokens of its block and all
// tokens of ancestor blocks; its rotary position is its position in its own
// prompt).  The long-request lane of "04 / Scheduling" runs a long row as
// several forwards, each resuming with the earlier tensors: here, chunks.
//
// Packing is depth-first pre-order, so the subtree of every block is one
// contiguous token interval [start, send); key j is then visible to query i
// exactly when j <= i < send[j].  Tiles of 128 queries x 128 keys are sorted
// into empty (dropped), full (no mask needed) and partial (per-element mask).

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <numeric>
#include <utility>

#include <cuda_runtime.h>

#include "internal.h"

namespace tree {

static thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

namespace {

constexpr int32_t kTile = 128;

size_t align4(size_t words) { return (words + 3) & ~size_t(3); }

// Bits [lo, hi) of a little-endian multi-word bit set, a word at a time.
void set_bits(int32_t *w, int32_t lo, int32_t hi) {
  while (lo < hi) {
    const int32_t k = lo >> 5, e = std::min(hi, (k + 1) << 5);
    const uint32_t n = (uint32_t)(e - lo);
    w[k] |= (int32_t)((n == 32 ? 0xffffffffu : ((1u << n) - 1u)) << (lo & 31));
    lo = e;
  }
}

// Bits [0, n) of a multi-word bit set all set.
bool all_bits(const int32_t *w, int32_t n) {
  for (int32_t k = 0; (k << 5) < n; ++k) {
    const int32_t m = std::min(32, n - (k << 5));
    const uint32_t want = m == 32 ? 0xffffffffu : ((1u << m) - 1u);
    if (((uint32_t)w[k] & want) != want) return false;
  }
  return true;
}

int build(const tree_spec_t &s, int32_t max_fwd, int32_t max_depth, int32_t max_row, int32_t tiling,
          int32_t pack_heads, Plan &P) {
  const int32_t nb = s.n_blocks;
  P.n_input_blocks = nb;
  P.max_fwd = max_fwd;
  P.tiling = tiling;
  P.pack_heads = pack_heads > 1 ? pack_heads : 1;
  // with R q heads packed per 128-row MMA tile, a query tile is two such tiles of 128 / R tokens
  P.bm = P.pack_heads > 1 ? 2 * (kTile / P.pack_heads) : kTile;
  const int32_t bm = P.bm;
  // ---- validation of the input forest
  for (int32_t b = 0; b < nb; ++b) {
    const int32_t p = s.parent[b];
    if (p < -1 || p >= nb || p == b)
      return fail(TREE_ERR_BAD_TREE, "block %d: parent %d out of range", b, p);
    if (s.length[b] <= 0) return fail(TREE_ERR_BAD_TREE, "block %d: length %d <= 0", b, s.length[b]);
  }
  // depth of every block by walking up; a chain longer than nb is a cycle
  std::vector<int32_t> depth(nb);
  int32_t dmax = 0;
  for (int32_t b = 0; b < nb; ++b) {
    int32_t d = 0;
    for (int32_t x = b; x != -1; x = s.parent[x]) {
      if (++d > nb) return fail(TREE_ERR_BAD_TREE, "block %d: parent chain has a cycle", b);
    }
    if (d > max_depth) return fail(TREE_ERR_DEPTH, "block %d: depth %d > %d", b, d, max_depth);
    depth[b] = d;
    dmax = std::max(dmax, d);
  }
  auto key_of = [&](int32_t b) -> uint64_t { return s.key ? s.key[b] : 0; };
  auto res_of = [&](int32_t b) -> int32_t { return s.resident ? (s.resident[b] ? 1 : 0) : 0; };

  // ---- merge identical siblings (trie semantics).  Blocks are visited by depth
  // and, within a depth, by input index, so a parent's merged identity is known
  // before its children and the first block of every identical group (the
  // lowest input index) becomes the group's block.  Two blocks are identical
  // when their merged parents, lengths and non-zero keys agree.
  std::vector<int32_t> by_depth(nb), dstart(dmax + 2, 0);
  for (int32_t b = 0; b < nb; ++b) ++dstart[depth[b] + 1];
  for (int32_t d = 1; d <= dmax + 1; ++d) dstart[d] += dstart[d - 1];
  {
    std::vector<int32_t> fill(dstart.begin(), dstart.end());
    for (int32_t b = 0; b < nb; ++b) by_depth[fill[depth[b]]++] = b;
  }
  std::vector<int32_t> canon(nb, -1), cparent(nb, -1);
  size_t cap = 16;
  while (cap < 2 * (size_t)nb) cap <<= 1;
  struct Slot {
    int32_t parent, len, block;
    uint64_t key;
  };
  std::vector<Slot> table(cap, Slot{0, 0, -1, 0});
  auto mix = [](uint64_t x) {
    x ^= x >> 33;
    x *= 0xff51afd7ed558ccdull;
    x ^= x >> 33;
    x *= 0xc4ceb9fe1a85ec53ull;
    return x ^ (x >> 33);
  };
  for (int32_t idx = 0; idx < nb; ++idx) {
    const int32_t b = by_depth[idx];
    const int32_t cp = s.parent[b] >= 0 ? canon[s.parent[b]] : -1;
    cparent[b] = cp;
    const uint64_t k = key_of(b);
    int32_t c = b;
    if (k != 0) {
      size_t h = mix(k ^ mix(((uint64_t)(uint32_t)cp << 32) | (uint32_t)s.length[b])) & (cap - 1);
      for (;; h = (h + 1) & (cap - 1)) {
        Slot &sl = table[h];
        if (sl.block < 0) {
          sl = Slot{cp, s.length[b], b, k};
          break;
        }
        if (sl.parent == cp && sl.len == s.length[b] && sl.key == k) {
          c = sl.block;
          break;
        }
      }
      if (c != b && res_of(b) != res_of(c))
        return fail(TREE_ERR_INVALID_ARG, "blocks %d and %d merge but disagree on residency", c, b);
    }
    canon[b] = c;
  }

  // ---- children of merged blocks (CSR, input order) and depth-first pre-order
  std::vector<int32_t> cstart(nb + 2, 0), clist;
  clist.reserve(nb);
  int32_t n_roots = 0;
  for (int32_t b = 0; b < nb; ++b) {
    if (canon[b] != b) continue;
    if (cparent[b] < 0)
      ++n_roots;
    else
      ++cstart[cparent[b] + 2];
  }
  for (int32_t i = 2; i <= nb + 1; ++i) cstart[i] += cstart[i - 1];
  clist.resize(cstart[nb + 1]);
  std::vector<int32_t> top;
  top.reserve(n_roots);
  for (int32_t b = 0; b < nb; ++b) {
    if (canon[b] != b) continue;
    if (cparent[b] < 0)
      top.push_back(b);
    else
      clist[cstart[cparent[b] + 1]++] = b;
  }
  // after the fill, cstart[c+1] is the end of c's children and cstart[c] their start
  std::vector<int32_t> packed;
  packed.reserve(nb);
  {
    std::vector<int32_t> st(top.rbegin(), top.rend());
    while (!st.empty()) {
      const int32_t c = st.back();
      st.pop_back();
      packed.push_back(c);
      for (int32_t i = cstart[c + 1] - 1; i >= cstart[c]; --i) st.push_back(clist[i]);
    }
  }
  const int32_t nbc = (int32_t)packed.size();
  P.n_blocks = nbc;
  std::vector<int32_t> pidx(nb, -1);
  for (int32_t i = 0; i < nbc; ++i) pidx[packed[i]] = i;
  P.block_map.resize(nb);
  for (int32_t b = 0; b < nb; ++b) P.block_map[b] = pidx[canon[b]];

  P.blk_start.assign(nbc, 0);
  P.blk_len.assign(nbc, 0);
  P.blk_parent.assign(nbc, -1);
  P.blk_depth.assign(nbc, 0);
  P.blk_pos0.assign(nbc, 0);
  P.blk_send.assign(nbc, 0);
  P.blk_resident.assign(nbc, 0);
  P.blk_slot.assign(nbc, -1);
  for (int32_t i = 0; i < nbc; ++i) {
    const int32_t c = packed[i];
    P.blk_len[i] = s.length[c];
    P.blk_parent[i] = s.parent[c] >= 0 ? pidx[canon[s.parent[c]]] : -1;
    P.blk_resident[i] = res_of(c);
  }
  std::vector<int64_t> sub(nbc);
  for (int32_t i = 0; i < nbc; ++i) {  // parents come first in pre-order
    const int32_t p = P.blk_parent[i];
    P.blk_depth[i] = p < 0 ? 1 : P.blk_depth[p] + 1;
    sub[i] = P.blk_len[i];
  }
  for (int32_t i = nbc - 1; i >= 0; --i)
    if (P.blk_parent[i] >= 0) sub[P.blk_parent[i]] += sub[i];
  int64_t tot = 0;
  for (int32_t i = 0; i < nbc; ++i) {
    if (P.blk_parent[i] < 0 && sub[i] > max_row)
      return fail(TREE_ERR_ROW_TOO_LONG, "row of %lld tokens > %d", (long long)sub[i], max_row);
    tot += P.blk_len[i];
  }
  if (tot > INT32_MAX / 2) return fail(TREE_ERR_INVALID_ARG, "%lld tokens: too many", (long long)tot);
  P.n_tot = (int32_t)tot;
  tot = 0;
  for (int32_t i = 0; i < nbc; ++i) {
    P.blk_start[i] = (int32_t)tot;
    tot += P.blk_len[i];
    const int32_t p = P.blk_parent[i];
    P.blk_pos0[i] = p < 0 ? 0 : P.blk_pos0[p] + P.blk_len[p];
    P.blk_send[i] = P.blk_start[i] + (int32_t)sub[i];
  }
  // ---- resident tokens lead the packed row
  int32_t n_res = 0;
  bool fwd_seen = false;
  for (int32_t i = 0; i < nbc; ++i) {
    if (P.blk_resident[i]) {
      if (fwd_seen)
        return fail(TREE_ERR_INVALID_ARG, "resident block %d follows a forward block in packed order", i);
      n_res += P.blk_len[i];
    } else {
      fwd_seen = true;
    }
  }
  if (n_res == P.n_tot) return fail(TREE_ERR_INVALID_ARG, "no forward tokens");
  P.n_res = n_res;

  const int32_t n_kvt = (P.n_tot + kTile - 1) / kTile;
  int32_t maxpos = 0;
  for (int32_t i = 0; i < nbc; ++i) maxpos = std::max(maxpos, P.blk_pos0[i] + P.blk_len[i]);
  P.max_pos = maxpos;
  const int32_t *bstart = P.blk_start.data(), *blen = P.blk_len.data(), *bpos0 = P.blk_pos0.data(),
                *bsend = P.blk_send.data();
  // packed block holding token t (blocks are sorted by start)
  auto block_of = [&](int32_t t) {
    return (int32_t)(std::upper_bound(P.blk_start.begin(), P.blk_start.end(), t) - P.blk_start.begin()) - 1;
  };
  // visible pairs of the queries in [a, b): each query sees pos + 1 keys
  auto pairs_in = [&](int32_t a, int32_t b) {
    int64_t sum = 0;
    for (int32_t i = block_of(a); i < nbc && bstart[i] < b; ++i) {
      const int64_t lo = std::max(a, bstart[i]), hi = std::min(b, bstart[i] + blen[i]);
      if (hi <= lo) continue;
      const int64_t first = bpos0[i] + (lo - bstart[i]) + 1;  // pos + 1 of token lo
      sum += (hi - lo) * first + (hi - lo) * (hi - lo - 1) / 2;
    }
    return sum;
  };
  P.pairs = pairs_in(P.n_res, P.n_tot);

  // per key tile: smallest and largest subtree end of its keys (padding keys count as 0)
  std::vector<int32_t> kt_min(n_kvt, INT32_MAX), kt_max(n_kvt, INT32_MIN);
  for (int32_t i = 0; i < nbc; ++i) {
    const int32_t k0 = bstart[i] / kTile, k1 = (bstart[i] + blen[i] - 1) / kTile;
    for (int32_t kt = k0; kt <= k1; ++kt) {
      kt_min[kt] = std::min(kt_min[kt], bsend[i]);
      kt_max[kt] = std::max(kt_max[kt], bsend[i]);
    }
  }
  if (P.n_tot % kTile) kt_min[n_kvt - 1] = 0;

  // ---- tiling by position: virtual key tiles.  For a query tile [i0, i1) and
  // position range t ([128t, 128t + 128)), every row takes the keys of its own
  // prompt in that range from exactly one entry, key at position p in slot
  // p % 128; entries follow in increasing t.  An entry gathers the keys of the
  // chain root -> d, d the deepest block of some row's chain that reaches into
  // the range; rows whose own such block is an ancestor of d ride along (their
  // keys of the range are a prefix of the entry's, in the same slots, and the
  // entry's other keys belong to blocks that are not their ancestors: not
  // visible to them).
  auto is_anc_or_self = [&](int32_t b, int32_t d) {
    for (int32_t x = d; x >= 0; x = P.blk_parent[x])
      if (x == b) return true;
    return false;
  };
  auto add_position_tiles = [&](int32_t i0, int32_t i1) {
    std::vector<int32_t> tb;  // blocks with rows in the tile, packed order
    for (int32_t b = block_of(i0); b < nbc && bstart[b] < i1; ++b)
      if (bstart[b] + blen[b] > i0) tb.push_back(b);
    auto pos_max = [&](int32_t b) { return bpos0[b] + (std::min(i1, bstart[b] + blen[b]) - 1 - bstart[b]); };
    int32_t tmax = 0;
    for (int32_t b : tb) tmax = std::max(tmax, pos_max(b) / kTile);
    std::vector<std::pair<int32_t, int32_t>> made;  // (entry, block) of this t
    for (int32_t t = 0; t <= tmax; ++t) {
      made.clear();
      for (size_t k = tb.size(); k-- > 0;) {
        const int32_t b = tb[k];
        if (pos_max(b) < t * kTile) continue;  // its rows see no key in this range
        // the deepest block of b's chain that reaches into the range: the keys of the
        // range on b's chain are those of the chain root -> db
        int32_t db = b;
        while (bpos0[db] >= (t + 1) * kTile) db = P.blk_parent[db];
        int32_t e = -1;
        for (const auto &m : made)
          if (is_anc_or_self(db, m.second)) {
            e = m.first;
            break;
          }
        if (e < 0) {
          e = (int32_t)P.ent.size();
          P.ent.push_back((e << 2) | 1);  // flags finished below, once every row is assigned
          const size_t kb = P.vkeys.size(), rb = P.vruns.size();
          P.vkeys.resize(kb + kTile, 0);
          P.vruns.resize(rb + kVRunWords, 0);
          // the chain root -> db, root first
          int32_t chain[64], nch = 0;
          for (int32_t x = db; x >= 0 && nch < 64; x = P.blk_parent[x]) chain[nch++] = x;
          int32_t n = 0;
          for (int32_t c = nch; c-- > 0;) {
            const int32_t blk = chain[c];
            const int32_t lo = std::max(bpos0[blk], t * kTile), hi = std::min(bpos0[blk] + blen[blk], (t + 1) * kTile);
            if (lo >= hi) continue;
            const int32_t c0 = lo - t * kTile, c1 = hi - 1 - t * kTile, j0 = bstart[blk] + (lo - bpos0[blk]);
            for (int32_t q = c0; q <= c1; ++q) P.vkeys[kb + q] = j0 + (q - c0);
            int32_t *run = P.vruns.data() + rb + 8 + 4 * n;
            run[0] = c0;
            run[1] = c1;
            run[2] = j0;
            run[3] = bsend[blk];
            ++n;
          }
          P.vruns[rb] = n;  // at most the depth of the tree (<= max_depth <= 16)
          made.emplace_back(e, db);
        }
        // the rows of b at positions >= 128 t take this range from entry e
        int32_t *rows = P.vruns.data() + (size_t)e * kVRunWords + 4;
        const int32_t r_lo = std::max(i0, bstart[b]), r_hi = std::min(i1, bstart[b] + blen[b]);
        const int32_t first = std::max(r_lo, bstart[b] + (t * kTile - bpos0[b]));
        set_bits(rows, first - i0, r_hi - i0);
      }
      // entries of this range: contiguous (slot c holds packed key j0 + c: one tiled load)
      // and full (every row of the tile is served by it and sees every slot: no mask)
      for (const auto &m : made) {
        const int32_t e = m.first;
        const int32_t *vk = P.vkeys.data() + (size_t)e * kTile;
        const int32_t *run = P.vruns.data() + (size_t)e * kVRunWords;
        const bool contig = run[0] == 1 && run[8] == 0 && run[9] == kTile - 1;
        bool full = contig && vk[kTile - 1] <= i0;
        if (full) {
          full = all_bits(run + 4, i1 - i0);  // every row of the tile is served by it
          full = full && run[11] > i1 - 1;
        }
        // a full contiguous entry needs neither its gather list nor its run table: it names
        // its first key instead, like a packed key tile
        P.ent[(size_t)e] = full ? ((vk[0] << 2) | 2) : ((e << 2) | (contig ? 2 : 0) | 1);
      }
    }
  };

  // ---- gathered key tiles (tiling 2).  A query sees every key of its ancestor
  // blocks and the keys of its own block up to itself, so the keys that some
  // query of the tile [i0, i1) sees are: each block with rows in the tile up to
  // its last row there, and the whole of every ancestor of those blocks.  They
  // fill entries of 128 slots in packed order, a run per piece of a block
  // (consecutive keys, one subtree end), at most kMaxRuns runs per entry.  A
  // run whose first key does not follow the previous run's last starts at a
  // slot that is a multiple of 8, so that the kernel loads each stretch of
  // consecutive keys as tiled boxes of 8k rows (the rows past a stretch's end
  // land in slots no run covers).
  std::vector<std::pair<int32_t, int32_t>> gathered;  // (block, key end), then merged per block
  auto add_gathered_tiles = [&](int32_t i0, int32_t i1) {
    gathered.clear();
    for (int32_t b = block_of(i0); b < nbc && bstart[b] < i1; ++b) {
      if (bstart[b] + blen[b] <= i0) continue;
      gathered.emplace_back(b, std::min(i1, bstart[b] + blen[b]));
      for (int32_t x = P.blk_parent[b]; x >= 0; x = P.blk_parent[x]) gathered.emplace_back(x, bstart[x] + blen[x]);
    }
    std::sort(gathered.begin(), gathered.end());
    int32_t e = -1, slot = kTile, nrun = kMaxRuns;
    size_t kb = 0, rb = 0;
    auto finish = [&]() {  // contiguous: every slot holds key (slot 0's key) + c; full: no mask at all
      if (e < 0) return;
      const int32_t *vk = P.vkeys.data() + kb, *run = P.vruns.data() + rb;
      bool contig = slot == kTile && run[0] > 0;
      for (int32_t c = 1; c < kTile && contig; ++c) contig = vk[c] == vk[0] + c;
      bool full = contig && vk[kTile - 1] <= i0;
      for (int32_t r = 0; r < run[0] && full; ++r) full = run[8 + 4 * r + 3] > i1 - 1;
      P.ent[(size_t)e] = full ? ((vk[0] << 2) | 2) : ((e << 2) | (contig ? 2 : 0) | 1);
    };
    for (size_t g = 0; g < gathered.size(); ++g) {
      const int32_t blk = gathered[g].first;
      int32_t end = gathered[g].second;
      while (g + 1 < gathered.size() && gathered[g + 1].first == blk) end = std::max(end, gathered[++g].second);
      int32_t j = bstart[blk];
      while (j < end) {
        if (nrun > 0 && slot < kTile) {
          const int32_t *prev = P.vruns.data() + rb + 8 + 4 * (nrun - 1);
          if (prev[2] + (prev[1] - prev[0]) + 1 != j) slot = (slot + 7) & ~7;  // a new stretch of keys
        }
        if (slot >= kTile || nrun == kMaxRuns) {
          finish();
          e = (int32_t)P.ent.size();
          P.ent.push_back(0);
          kb = P.vkeys.size();
          rb = P.vruns.size();
          P.vkeys.resize(kb + kTile, 0);
          P.vruns.resize(rb + kVRunWords, 0);
          set_bits(P.vruns.data() + rb + 4, 0, i1 - i0);  // every row of the tile takes every entry
          slot = 0;
          nrun = 0;
        }
        const int32_t n = std::min(end - j, kTile - slot);
        for (int32_t c = 0; c < n; ++c) P.vkeys[kb + slot + c] = j + c;
        int32_t *run = P.vruns.data() + rb + 8 + 4 * nrun;
        run[0] = slot;
        run[1] = slot + n - 1;
        run[2] = j;
        run[3] = bsend[blk];
        P.vruns[rb] = ++nrun;
        slot += n;
        j += n;
      }
    }
    finish();
  };

  // ---- chunks, query tiles, tile lists
  const int32_t n_fwd = P.n_tot - P.n_res;
  P.n_chunks = (n_fwd + max_fwd - 1) / max_fwd;
  const int32_t n_qt_est = (n_fwd + bm - 1) / bm + P.n_chunks;
  P.qt_row0.reserve(n_qt_est);
  P.qt_row1.reserve(n_qt_est);
  P.qt_ent0.reserve(n_qt_est);
  P.qt_ent1.reserve(n_qt_est);
  P.qt_order.reserve(n_qt_est);
  P.ent.reserve((size_t)n_qt_est * 8);
  if (tiling == 1) {
    // an upper bound on the entries (per query tile: position ranges x blocks with rows in
    // it), so the gather lists and run tables are allocated once
    size_t bound = 0;
    for (int32_t c = 0; c < P.n_chunks; ++c) {
      const int32_t q0 = P.n_res + c * max_fwd, q1 = std::min(q0 + max_fwd, P.n_tot);
      for (int32_t i0 = q0; i0 < q1; i0 += kTile) {
        const int32_t i1 = std::min(i0 + kTile, q1);
        int32_t nblk = 0, tmax = 0;
        for (int32_t b = block_of(i0); b < nbc && bstart[b] < i1; ++b) {
          if (bstart[b] + blen[b] <= i0) continue;
          ++nblk;
          tmax = std::max(tmax, (bpos0[b] + (std::min(i1, bstart[b] + blen[b]) - 1 - bstart[b])) / kTile);
        }
        bound += (size_t)(tmax + 1) * nblk;
      }
    }
    P.ent.reserve(P.ent.size() + bound);
    P.vkeys.reserve(bound * kTile);
    P.vruns.reserve(bound * kVRunWords);
  }
  std::vector<int32_t> ord;
  for (int32_t c = 0; c < P.n_chunks; ++c) {
    const int32_t q0 = P.n_res + c * max_fwd, q1 = std::min(q0 + max_fwd, P.n_tot);
    P.chunk_q0.push_back(q0);
    P.chunk_q1.push_back(q1);
    P.chunk_t0.push_back((int32_t)P.qt_row0.size());
    P.chunk_pairs.push_back(pairs_in(q0, q1));
    const int32_t e_begin = (int32_t)P.ent.size();
    for (int32_t i0 = q0; i0 < q1; i0 += bm) {
      const int32_t i1 = std::min(i0 + bm, q1);
      P.qt_row0.push_back(i0);
      P.qt_row1.push_back(i1);
      P.qt_ent0.push_back((int32_t)P.ent.size());
      if (tiling == 1) {
        add_position_tiles(i0, i1);
        P.qt_ent1.push_back((int32_t)P.ent.size());
        continue;
      }
      if (tiling == 2) {
        add_gathered_tiles(i0, i1);
        P.qt_ent1.push_back((int32_t)P.ent.size());
        continue;
      }
      const int32_t last = (i1 - 1) / kTile;
      for (int32_t kt = 0; kt <= last; ++kt) {
        const int32_t j0 = kt * kTile, j1 = j0 + kTile;
        // some query sees some key: a key j < i1 whose subtree reaches past i0
        bool any;
        if (j1 <= i1) {
          any = kt_max[kt] > i0;
        } else {
          any = false;
          for (int32_t i = block_of(j0); i < nbc && bstart[i] < i1 && !any; ++i) any = bsend[i] > i0;
        }
        if (!any) continue;
        // every query sees every key: the tile is whole, lies before the
        // first query, and every key's subtree reaches past the last query
        const bool full = (j1 <= P.n_tot) && (j1 - 1 <= i0) && (i1 - 1 < kt_min[kt]);
        P.ent.push_back((kt << 1) | (full ? 0 : 1));
      }
      P.qt_ent1.push_back((int32_t)P.ent.size());
    }
    P.chunk_t1.push_back((int32_t)P.qt_row0.size());
    P.chunk_nent.push_back((int32_t)P.ent.size() - e_begin);
    // longest-first order of the chunk's tiles; equal work keeps tile order
    ord.resize(P.chunk_t1[c] - P.chunk_t0[c]);
    std::iota(ord.begin(), ord.end(), P.chunk_t0[c]);
    std::stable_sort(ord.begin(), ord.end(), [&](int32_t a, int32_t b) {
      return P.qt_ent1[a] - P.qt_ent0[a] > P.qt_ent1[b] - P.qt_ent0[b];
    });
    P.qt_order.insert(P.qt_order.end(), ord.begin(), ord.end());
  }

  // ---- readout slots: last token of every leaf, packed order
  std::vector<char> has_child(nbc, 0);
  for (int32_t i = 0; i < nbc; ++i)
    if (P.blk_parent[i] >= 0) has_child[P.blk_parent[i]] = 1;
  for (int32_t i = 0; i < nbc; ++i) {
    if (has_child[i]) continue;
    P.blk_slot[i] = (int32_t)P.slot_tok.size();
    P.slot_tok.push_back(P.blk_start[i] + P.blk_len[i] - 1);
  }
  P.n_questions = s.n_questions;
  for (int32_t q = 0; q < s.n_questions; ++q) {
    const int32_t l[2] = {s.leaf1[q], s.leaf2[q]};
    for (int32_t o = 0; o < 2; ++o) {
      if (l[o] < 0 || l[o] >= nb) return fail(TREE_ERR_INVALID_ARG, "question %d: block %d out of range", q, l[o]);
      const int32_t slot = P.blk_slot[P.block_map[l[o]]];
      if (slot < 0) return fail(TREE_ERR_INVALID_ARG, "question %d: block %d is not a leaf", q, l[o]);
      (o == 0 ? P.r1 : P.r2).push_back(slot);
    }
  }

  // ---- device image; the per-token tables are written into it directly
  const size_t n_send = (size_t)n_kvt * kTile;
  size_t w = 16;  // header words
  P.off_pos = w;
  w = align4(w + P.n_tot);
  P.off_send = w;
  w = align4(w + n_send);
  P.off_qtile = w;
  w = align4(w + 4 * P.qt_row0.size());
  P.off_ent = w;
  w = align4(w + P.ent.size());
  P.off_order = w;
  w = align4(w + P.qt_order.size());
  P.off_chunk = w;
  w = align4(w + 4 * (size_t)P.n_chunks);
  P.off_slot_tok = w;
  w = align4(w + P.slot_tok.size());
  P.off_r1 = w;
  w = align4(w + P.r1.size());
  P.off_r2 = w;
  w = align4(w + P.r2.size());
  P.off_runs = w;
  w = align4(w + (size_t)n_kvt * kRunWords);
  P.off_vkeys = w;
  w = align4(w + P.vkeys.size());
  P.off_vruns = w;
  w = align4(w + P.vruns.size());
  P.image.resize(w);
  int32_t *im = P.image.data();
  std::fill(im, im + 16, 0);
  im[0] = 0x4C505254;  // "TRPL"
  im[1] = P.n_tot;
  im[2] = P.n_res;
  im[3] = P.n_chunks;
  im[4] = (int32_t)P.qt_row0.size();
  im[5] = (int32_t)P.ent.size();
  im[6] = (int32_t)P.slot_tok.size();
  im[7] = P.n_questions;
  int32_t *pos = im + P.off_pos, *send = im + P.off_send;
  for (int32_t i = 0; i < nbc; ++i) {  // two plain fills per block (each vectorises on its own)
    const int32_t st = bstart[i], len = blen[i], p0 = bpos0[i];
    int32_t *pp = pos + st;
    for (int32_t t = 0; t < len; ++t) pp[t] = p0 + t;
    std::fill(send + st, send + st + len, bsend[i]);
  }
  std::fill(send + P.n_tot, send + n_send, 0);
  for (size_t t = 0; t < P.qt_row0.size(); ++t) {
    int32_t *r = im + P.off_qtile + 4 * t;
    r[0] = P.qt_row0[t];
    r[1] = P.qt_row1[t];
    r[2] = P.qt_ent0[t];
    r[3] = P.qt_ent1[t];
  }
  std::copy(P.ent.begin(), P.ent.end(), im + P.off_ent);
  std::copy(P.qt_order.begin(), P.qt_order.end(), im + P.off_order);
  for (int32_t c = 0; c < P.n_chunks; ++c) {
    int32_t *r = im + P.off_chunk + 4 * c;
    r[0] = P.chunk_q0[c];
    r[1] = P.chunk_q1[c];
    r[2] = P.chunk_t0[c];
    r[3] = P.chunk_t1[c];
  }
  std::copy(P.slot_tok.begin(), P.slot_tok.end(), im + P.off_slot_tok);
  std::copy(P.r1.begin(), P.r1.end(), im + P.off_r1);
  std::copy(P.r2.begin(), P.r2.end(), im + P.off_r2);
  // run tables of the key tiles: maximal runs of equal send.  A tile's keys fall
  // into a few block segments of constant send (padding past the last token:
  // send 0), so the runs are built segment by segment.
  std::fill(im + P.off_runs, im + P.off_runs + (size_t)n_kvt * kRunWords, 0);
  {
    int32_t b = 0;  // first block that ends after the tile's first key
    for (int32_t t = 0; t < n_kvt; ++t) {
      int32_t *tb = im + P.off_runs + (size_t)t * kRunWords;
      const int32_t j0 = t * kTile, j1 = j0 + kTile;
      while (b < nbc && bstart[b] + blen[b] <= j0) ++b;
      int32_t n = 0, last = 0;
      auto segment = [&](int32_t lo, int32_t hi, int32_t value) {  // keys [lo, hi) of the tile
        if (n == 0 || value != last) {
          if (n < kMaxRuns) tb[4 + n] = value;
          ++n;
          last = value;
        }
        if (n > kMaxRuns) return;
        int32_t *bits = tb + 20 + 4 * (n - 1);
        for (int32_t c = lo - j0; c < hi - j0;) {  // set bits c .. (word end or hi) at once
          const int32_t wd = c >> 5, e = std::min(hi - j0, (wd + 1) << 5);
          const uint32_t lo_bit = (uint32_t)(c & 31), cnt = (uint32_t)(e - c);
          bits[wd] |= (int32_t)((cnt == 32 ? 0xffffffffu : ((1u << cnt) - 1u)) << lo_bit);
          c = e;
        }
      };
      for (int32_t i = b; i < nbc && bstart[i] < j1; ++i)
        segment(std::max(j0, bstart[i]), std::min(j1, bstart[i] + blen[i]), bsend[i]);
      if (j1 > P.n_tot) segment(std::max(j0, P.n_tot), j1, 0);
      tb[0] = n;
      if (n > kMaxRuns) std::fill(tb + 4, tb + kRunWords, 0);  // only the count is meaningful
    }
  }
  // zero the alignment gaps so the image is fully defined
  auto zero_gap = [&](size_t from, size_t to) { std::fill(im + from, im + to, 0); };
  zero_gap(P.off_pos + P.n_tot, P.off_send);
  zero_gap(P.off_qtile + 4 * P.qt_row0.size(), P.off_ent);
  zero_gap(P.off_ent + P.ent.size(), P.off_order);
  zero_gap(P.off_order + P.qt_order.size(), P.off_chunk);
  zero_gap(P.off_chunk + 4 * (size_t)P.n_chunks, P.off_slot_tok);
  zero_gap(P.off_slot_tok + P.slot_tok.size(), P.off_r1);
  zero_gap(P.off_r1 + P.r1.size(), P.off_r2);
  zero_gap(P.off_r2 + P.r2.size(), P.off_runs);
  std::copy(P.vkeys.begin(), P.vkeys.end(), im + P.off_vkeys);
  std::copy(P.vruns.begin(), P.vruns.end(), im + P.off_vruns);
  zero_gap(P.off_runs + (size_t)n_kvt * kRunWords, P.off_vkeys);
  zero_gap(P.off_vkeys + P.vkeys.size(), P.off_vruns);
  zero_gap(P.off_vruns + P.vruns.size(), w);
  return TREE_OK;
}

// The largest buffers of the plans freed on this thread, kept for the next plan
// built here: a runtime plans batch after batch, and fresh multi-megabyte
// buffers would cost a page fault per page every time.
struct Spare {
  std::vector<int32_t> image, vkeys, vruns;
};
thread_local Spare g_spare;

void keep_larger(std::vector<int32_t> &spare, std::vector<int32_t> &v) {
  if (v.capacity() > spare.capacity()) spare.swap(v);
}

void take_spare(Plan &P) {
  P.image.swap(g_spare.image);
  P.vkeys.swap(g_spare.vkeys);
  P.vruns.swap(g_spare.vruns);
  P.image.clear();
  P.vkeys.clear();
  P.vruns.clear();
}

void give_spare(Plan &P) {
  keep_larger(g_spare.image, P.image);
  keep_larger(g_spare.vkeys, P.vkeys);
  keep_larger(g_spare.vruns, P.vruns);
}

}  // namespace
}  // namespace tree

extern "C" {

const char *tree_last_error(void) { return tree::g_err.c_str(); }

int tree_version(void) { return 101; }

int tree_pack_plan(const tree_spec_t *spec, const tree_plan_opts_t *opts, tree_plan_t **out) {
  if (!spec || !out) return tree::fail(TREE_ERR_INVALID_ARG, "tree_pack_plan: NULL spec or out");
  *out = nullptr;
  if (spec->n_blocks <= 0 || !spec->parent || !spec->length)
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_pack_plan: empty forest or NULL parent/length");
  if (spec->n_questions < 0 || (spec->n_questions > 0 && (!spec->leaf1 || !spec->leaf2)))
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_pack_plan: bad question arrays");
  int32_t max_fwd = 8192, max_depth = 8, max_row = 32768, tiling = 0, pack_heads = 0;
  if (opts) {
    if (opts->max_fwd) max_fwd = opts->max_fwd;
    if (opts->max_depth) max_depth = opts->max_depth;
    if (opts->max_row) max_row = opts->max_row;
    tiling = opts->tiling;
    pack_heads = opts->pack_heads;
  }
  if (max_fwd <= 0 || max_fwd % 128 != 0)
    return tree::fail(TREE_ERR_UNSUPPORTED, "max_fwd %d is not a positive multiple of 128", max_fwd);
  if (max_depth <= 0 || max_row <= 0) return tree::fail(TREE_ERR_INVALID_ARG, "bad limits");
  if (tiling < 0 || tiling > 2) return tree::fail(TREE_ERR_INVALID_ARG, "tiling %d is not 0, 1 or 2", tiling);
  if (pack_heads < 0 || pack_heads > 8 || (pack_heads & (pack_heads - 1)))
    return tree::fail(TREE_ERR_INVALID_ARG, "pack_heads %d is not 0, 1, 2, 4 or 8", pack_heads);
  if (pack_heads > 1 && tiling == 0)
    return tree::fail(TREE_ERR_UNSUPPORTED, "pack_heads %d needs key tiles by position or gathered (tiling 1, 2)",
                      pack_heads);
  if (tiling == 1 && max_depth > tree::kMaxRuns)
    return tree::fail(TREE_ERR_UNSUPPORTED, "tiling by position needs max_depth <= %d", tree::kMaxRuns);
  auto *pl = new (std::nothrow) tree_plan;
  if (!pl) return tree::fail(TREE_ERR_INVALID_ARG, "out of host memory");
  tree::take_spare(pl->p);
  const int rc = tree::build(*spec, max_fwd, max_depth, max_row, tiling, pack_heads, pl->p);
  if (rc != TREE_OK) {
    tree::give_spare(pl->p);
    delete pl;
    return rc;
  }
  *out = pl;
  return TREE_OK;
}

int tree_plan_free(tree_plan_t *plan) {
  if (plan) tree::give_spare(plan->p);
  delete plan;
  return TREE_OK;
}

int tree_plan_query(const tree_plan_t *plan, tree_plan_info_t *info) {
  if (!plan || !info) return tree::fail(TREE_ERR_INVALID_ARG, "tree_plan_query: NULL argument");
  const tree::Plan &P = plan->p;
  std::memset(info, 0, sizeof *info);
  info->n_input_blocks = P.n_input_blocks;
  info->n_blocks = P.n_blocks;
  info->n_tot = P.n_tot;
  info->n_res = P.n_res;
  info->n_fwd = P.n_tot - P.n_res;
  info->n_chunks = P.n_chunks;
  info->n_qtiles = (int32_t)P.qt_row0.size();
  info->n_entries = (int32_t)P.ent.size();
  info->n_slots = (int32_t)P.slot_tok.size();
  info->n_questions = P.n_questions;
  info->max_fwd = P.max_fwd;
  info->bm = P.bm;
  info->bn = P.bn;
  info->max_pos = P.max_pos;
  info->pairs = P.pairs;
  info->dev_bytes = P.image.size() * sizeof(int32_t);
  info->off_pos = P.off_pos * 4;
  info->off_send = P.off_send * 4;
  info->off_qtile = P.off_qtile * 4;
  info->off_ent = P.off_ent * 4;
  info->off_order = P.off_order * 4;
  info->off_chunk = P.off_chunk * 4;
  info->off_slot_tok = P.off_slot_tok * 4;
  info->off_r1 = P.off_r1 * 4;
  info->off_r2 = P.off_r2 * 4;
  info->off_runs = P.off_runs * 4;
  info->tiling = P.tiling;
  info->off_vkeys = P.off_vkeys * 4;
  info->off_vruns = P.off_vruns * 4;
  info->pack_heads = P.pack_heads;
  return TREE_OK;
}

int tree_plan_chunk(const tree_plan_t *plan, int32_t chunk, tree_chunk_info_t *info) {
  if (!plan || !info) return tree::fail(TREE_ERR_INVALID_ARG, "tree_plan_chunk: NULL argument");
  const tree::Plan &P = plan->p;
  if (chunk < 0 || chunk >= P.n_chunks)
    return tree::fail(TREE_ERR_INVALID_ARG, "chunk %d out of range [0, %d)", chunk, P.n_chunks);
  info->q0 = P.chunk_q0[chunk];
  info->q1 = P.chunk_q1[chunk];
  info->t0 = P.chunk_t0[chunk];
  info->t1 = P.chunk_t1[chunk];
  info->pairs = P.chunk_pairs[chunk];
  info->n_entries = P.chunk_nent[chunk];
  return TREE_OK;
}

int tree_plan_tables(const tree_plan_t *plan, tree_plan_host_view_t *v) {
  if (!plan || !v) return tree::fail(TREE_ERR_INVALID_ARG, "tree_plan_tables: NULL argument");
  const tree::Plan &P = plan->p;
  v->block_map = P.block_map.data();
  v->blk_start = P.blk_start.data();
  v->blk_len = P.blk_len.data();
  v->blk_parent = P.blk_parent.data();
  v->blk_depth = P.blk_depth.data();
  v->blk_pos0 = P.blk_pos0.data();
  v->blk_send = P.blk_send.data();
  v->blk_resident = P.blk_resident.data();
  v->blk_slot = P.blk_slot.data();
  v->pos = P.image.data() + P.off_pos;
  v->send = P.image.data() + P.off_send;
  v->runs = P.image.data() + P.off_runs;
  v->vkeys = P.tiling != 0 ? P.image.data() + P.off_vkeys : nullptr;
  v->vruns = P.tiling != 0 ? P.image.data() + P.off_vruns : nullptr;
  v->chunk_q0 = P.chunk_q0.data();
  v->chunk_q1 = P.chunk_q1.data();
  v->chunk_t0 = P.chunk_t0.data();
  v->chunk_t1 = P.chunk_t1.data();
  v->qt_row0 = P.qt_row0.data();
  v->qt_row1 = P.qt_row1.data();
  v->qt_ent0 = P.qt_ent0.data();
  v->qt_ent1 = P.qt_ent1.data();
  v->ent = P.ent.data();
  v->qt_order = P.qt_order.data();
  v->slot_tok = P.slot_tok.data();
  v->r1 = P.r1.data();
  v->r2 = P.r2.data();
  v->image = P.image.data();
  v->image_bytes = P.image.size() * sizeof(int32_t);
  return TREE_OK;
}

int tree_plan_upload(const tree_plan_t *plan, void *dev_buf, size_t bytes, tree_stream_t stream) {
  if (!plan || !dev_buf) return tree::fail(TREE_ERR_INVALID_ARG, "tree_plan_upload: NULL argument");
  const size_t need = plan->p.image.size() * sizeof(int32_t);
  if (bytes < need)
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_plan_upload: buffer of %zu bytes < %zu", bytes, need);
  if (reinterpret_cast<uintptr_t>(dev_buf) % 16)
    return tree::fail(TREE_ERR_UNSUPPORTED, "tree_plan_upload: device buffer not 16-byte aligned");
  const cudaError_t e = cudaMemcpyAsync(dev_buf, plan->p.image.data(), need, cudaMemcpyHostToDevice,
                                        reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return tree::fail(TREE_ERR_CUDA, "tree_plan_upload: %s", cudaGetErrorString(e));
  return TREE_OK;
}

int tree_plan_upload_staged(const tree_plan_t *plan, void *dev_buf, size_t bytes, void *host_staging,
                            size_t staging_bytes, tree_stream_t stream) {
  if (!plan || !dev_buf || !host_staging)
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_plan_upload_staged: NULL argument");
  const size_t need = plan->p.image.size() * sizeof(int32_t);
  if (bytes < need || staging_bytes < need)
    return tree::fail(TREE_ERR_INVALID_ARG, "tree_plan_upload_staged: buffers of %zu / %zu bytes < %zu", bytes,
                      staging_bytes, need);
  if (reinterpret_cast<uintptr_t>(dev_buf) % 16)
    return tree::fail(TREE_ERR_UNSUPPORTED, "tree_plan_upload_staged: device buffer not 16-byte aligned");
  std::memcpy(host_staging, plan->p.image.data(), need);
  const cudaError_t e = cudaMemcpyAsync(dev_buf, host_staging, need, cudaMemcpyHostToDevice,
                                        reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return tree::fail(TREE_ERR_CUDA, "tree_plan_upload_staged: %s", cudaGetErrorString(e));
  return TREE_OK;
}

}  // extern "C"
