// Pieces shared by the tree-attention kernels: launch arguments, bounded
// mbarrier waits and the work-item decoding (one query tile, one kv head, a
// group of the q heads that read it).
#pragma once

#include "common.cuh"
#include "sm103.cuh"

namespace tree {
namespace attn {

using namespace sm103;

constexpr int BN = 128;                    // keys per tile (queries per tile: 128, one per TMEM lane)
constexpr uint32_t BOX_BYTES = 128 * 128;  // one 128-row x 64-column f16 box (128-byte rows)
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 500000000ull;
constexpr uint64_t kSelfTestNs = 2000000ull;

struct AttnArgs {
  const int32_t *send;
  const int32_t *runs;  // run tables of the key tiles
  const int32_t *vkeys, *vruns;  // tiling by position: each entry's gathered keys and run table
  const QTile *qtiles;
  const int32_t *ent;
  const int32_t *order;
  __half *o;
  float *lse;
  int32_t *status;
  int32_t t0, q0, n_tot, hq, hkv, ratio;
  int32_t n_items;  // query tiles of the chunk x kv heads x q-head groups
  int32_t *work;    // {next item, finished CTAs} or nullptr for the round-robin schedule
  float scale_log2;
  int32_t self_test;  // the timeout self-test (see tree_attn_params_t)
  int32_t tpm;        // packed heads: tokens per 128-row MMA tile (128 / q heads per kv head)
  int32_t boxes;      // gathered tiles (tiling 2): runs load as tiled boxes of 8k rows, not row by row
};

// Tiling 2: maps of K and V with boxes of 8, 16, 32 and 64 rows (64 columns).
struct BoxMaps {
  CUtensorMap k[4], v[4];
};

constexpr int kRing = 4;  // items handed from the producer to the MMA and softmax warps

// Wait for the phase with the given parity; false (and the CTA's abort flag
// set) if it has not completed within limit_ns, or, with honor_abort, as soon
// as another thread of the CTA has given up.
TREE_DEV bool wait_bar(uint32_t bar, uint32_t parity, volatile int32_t *abort, int32_t *status,
                       bool honor_abort = true, uint64_t limit_ns = kWaitNs) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    // try_wait's default suspend window: measured faster than longer sleeps
    // (a long hint delays the wake-up after the phase completes)
    if (mbar_try(bar, parity)) return true;
    if ((n & 255) == 0) {
      if (honor_abort && *abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        if (status) atomicExch(status, TREE_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Warp-uniform form: the caller's next steps are warp-collective.  Every lane
// polls (measured faster than one polling lane plus a broadcast).
TREE_DEV bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int32_t *abort, int32_t *status) {
  const bool ok = wait_bar(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok);
}

// One work item: a query tile, the kv head g, and the NH q heads h0.. that read it.
struct Item {
  QTile qt;
  int n;   // key tiles in its list
  int h0;  // first q head
  int g;   // kv head
};

// With packed heads (HP) an item is a query tile and one kv head, and h0 is the
// first of all ratio q heads that read it (the MMA tiles hold every q head).
template <int NH, bool HP = false>
TREE_DEV Item item_at(const AttnArgs &a, int w) {
  const int groups = HP ? 1 : a.ratio / NH;
  const int per_tile = a.hkv * groups;
  const int rank = w / per_tile;
  const int rem = w - rank * per_tile;
  Item it;
  it.g = rem / groups;
  it.h0 = it.g * a.ratio + (rem - it.g * groups) * NH;
  it.qt = a.qtiles[__ldg(a.order + a.t0 + rank)];
  it.n = it.qt.ent1 - it.qt.ent0;
  return it;
}

}  // namespace attn

}  // namespace tree
