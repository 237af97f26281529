// tree_attn_fwd: attention over tree blocks for one forward chunk, sm_103a.
//
// A token sees the earlier tokens of its own block and every token of its
// ancestor blocks; sibling branches are masked, so each prompt's result equals
// computing it alone (basal-rs Architecture page, "03 / Packing: Attention
// over tree blocks").  With the planner's depth-first packing, key j is visible
// to query i iff j <= i < send[j].  Scores q.k * scale with scale = 1/sqrt(d)
// (AstrAI inference page, "KV Cache"); f16 storage, f32 softmax and
// accumulation ("01 / Request path: GPU forward pass").
//
// Work decomposition.  One CTA per (128-row query tile, kv head, pair of q
// heads that share that kv head); CTAs are ordered longest tile first from the
// planner's per-chunk order.  The CTA walks the tile's list of 128-key tiles
// (empty tiles never appear in it); full tiles skip the mask, partial tiles
// apply j <= i < send[j] per element.  Each K/V tile is loaded once and serves
// both q heads.
//
// Roles (warp specialisation, 12 warps for two heads):
//   softmax warpgroup h (warps 4h..4h+3), one per q head: thread = query row.
//       Reads its whole S row (128 f32) from tensor memory in one pass, masks,
//       keeps a running max and sum in the log2 domain, writes P (f16) to
//       tensor memory, and rescales O in tensor memory only when the running
//       max grows by more than 2^8 (rare); at the end normalises O and stores
//       it.  At d = 64 these warps raise their register budget to 208 (setmaxnreg).
//   producer warp: TMA loads of the Q tiles and of K, V (plus the 128 subtree
//       ends of the key tile) into a ring of shared-memory stages.
//   MMA warp: one thread issues tcgen05.mma: S_h = Q_h K^T (A, B in shared
//       memory, 128 x 128 x d) and O_h += P_h V (A = P_h in tensor memory,
//       B = V in shared memory, 128 x d x 128), each followed by a commit to an
//       mbarrier.  At d = 64 the producer/MMA warpgroup lowers its budget to 88 registers.
// Tensor memory (512 columns for two heads):
//   d = 64 : S_h at 128h, P_h at 256 + 64h, O_h at 384 + 64h.  S_h is free as
//            soon as the softmax has read it, so S_h(i+1) is computed while the
//            softmax still works on tile i.
//   d = 128: S_h at 128h with P_h over its first 64 columns, O_h at 256 + 128h;
//            S_h(i+1) waits until PV_h(i) has read P_h, and the two heads'
//            chains interleave on the tensor core.
//
// Every wait on an mbarrier gives up after ~2 s, sets TREE_ERR_TIMEOUT in the
// caller's status word, and the CTA winds down: pending copies and MMAs are
// awaited (bounded), tensor memory is freed, and the kernel returns.

#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "attn_common.cuh"

namespace tree {
namespace {

using namespace sm103;
using namespace attn;

template <int D, int NH>
struct Cfg {
  static constexpr int CB = D / 64;               // 64-column boxes per row of a tile
  static constexpr int STAGES = D == 64 ? 3 : 2;  // K/V ring depth
  static constexpr int QBUF = D == 64 ? 2 : 1;    // Q tiles in flight (next item's Q loads early)
  static constexpr uint32_t Q_BYTES = NH * CB * BOX_BYTES;
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + QBUF * Q_BYTES;
  static constexpr uint32_t V_OFF = K_OFF + STAGES * CB * BOX_BYTES;
  static constexpr uint32_t O_OFF = V_OFF + STAGES * CB * BOX_BYTES;  // per head: one 128 x 64 staging box
  static constexpr uint32_t RUNS_OFF = O_OFF + NH * BOX_BYTES;       // per stage: the key tile's run table
  static constexpr uint32_t SMEM = RUNS_OFF + STAGES * 512 + 1024;  // + alignment slack
  static constexpr int WARPS = 4 * NH + 4;        // softmax warpgroups + producer/MMA warpgroup
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int PROD_WARP = 4 * NH;
  static constexpr int MMA_WARP = 4 * NH + 1;    // MMA warps MMA_WARP .. MMA_WARP + MW - 1
  static constexpr int MW = D == 64 ? NH : 1;     // MMA warps: one per head at d = 64, one at d = 128
  static constexpr bool KV_ONE = STAGES >= 3;     // K and V of a stage complete one barrier
  // At d = 64 the two heads' softmax warps that share an SM sub-partition take
  // turns at the arithmetic of a tile (head 0, head 1, head 0, ...): the
  // arithmetic is issue-bound, so while one head computes, the other waits on
  // tensor memory and barriers instead of competing for the same issue slots.
  static constexpr bool ALT = NH == 2 && D == 64;
  static constexpr bool PSEP = D == 64;           // P in its own columns
  // d = 128: an item's epilogue waits until the next item's first P is stored
  // (measured faster there; at d = 64 it delays the next item's first PV)
  static constexpr bool DEFER = !PSEP;
  static constexpr uint32_t P_COL = 128 * NH;     // P_h at P_COL + 64h (PSEP only)
  static constexpr uint32_t O_COL = PSEP ? 128 * NH + 64 * NH : 128 * NH;
  static constexpr uint32_t TMEM_USED = O_COL + D * NH;
  static constexpr uint32_t TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
  // 12 warps launch at 168 registers (3 per SM sub-partition of 16384); at d = 64 setmaxnreg
  // moves them from the producer/MMA warpgroup to the softmax warpgroups.  An increase draws
  // only on what the block launched with, so the shares must add up to no more than that: a
  // larger sum makes setmaxnreg.inc wait forever.  The d = 128 instances keep 168 in every
  // warp: under a split, some of them computed wrong results, and which one did changed with
  // the shares (208/88, 200/104) and the number of MMA warps.
  static constexpr bool SPLIT = NH == 2 && D == 64;
  static constexpr int LAUNCH_REGS = 168;
  static constexpr int SOFTMAX_REGS = 208;
  static constexpr int SERVICE_REGS = 88;
  static_assert(!SPLIT || 128 * (NH * SOFTMAX_REGS + SERVICE_REGS) <= THREADS * LAUNCH_REGS,
                "register split exceeds the block's launch allotment");
};


struct Bars {
  uint64_t item_full[kRing], item_empty[kRing];
  int32_t ring[kRing][8];  // claimed item: {w, row0, row1, ent0, ent1, h0, g, first entry}
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[3], v_full[3], kv_empty[3];
  uint64_t s_full[2], s_free[2], p_full[2], o_done[2], o_free[2];
  uint64_t ostage_full[2], ostage_free[2];  // output staging box of each head
  uint64_t turn[2][4];  // per lane quarter: head h's warp has finished the arithmetic of its tile
  uint64_t never;  // a barrier nothing arrives on (timeout self-test)
  uint32_t tmem;
  int32_t abort;
};


// Persistent CTAs (one per SM).  The producer warp takes items from the
// longest-first item list -- with a work counter, the next unclaimed item as the
// CTA frees up; without one, items c, c + G, c + 2G, ... (G = grid size) -- and
// hands them to the MMA and softmax warps through a small ring in shared memory.
// Tiles are numbered across the CTA's items in the order it processes them;
// every barrier phase follows that count (or the item count for per-item
// barriers), so the producer and MMA warps run ahead into the next item while
// the softmax warps finish the current one.
// HP (packed heads, with gathered key tiles): the item is a query tile of 2 x tpm
// tokens and one kv head; MMA tile h holds tokens [row0 + h tpm, row0 + (h+1) tpm)
// of all ratio = 128 / tpm q heads (row r: head h0 + r / tpm, token r % tpm), so
// the item's K/V tiles serve every q head of the kv head at once.
template <int D, int NH, bool G, bool HP>
__global__ void __launch_bounds__(Cfg<D, NH>::THREADS, 1)
    tree_attn_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mo,
                 const __grid_constant__ CUtensorMap mkg, const __grid_constant__ CUtensorMap mvg,
                 const __grid_constant__ BoxMaps bm, const AttnArgs a) {
  using C = Cfg<D, NH>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(sm);
  const int32_t *sRuns = reinterpret_cast<const int32_t *>(sm + C::RUNS_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int32_t *abort = &bars.abort;

  auto b_if = [&](int r) { return smem_u32(&bars.item_full[r]); };
  auto b_ie = [&](int r) { return smem_u32(&bars.item_empty[r]); };
  auto b_qf = [&](int b) { return smem_u32(&bars.q_full[b]); };
  auto b_qe = [&](int b) { return smem_u32(&bars.q_empty[b]); };
  auto b_k = [&](int s) { return smem_u32(&bars.k_full[s]); };
  auto b_v = [&](int s) { return smem_u32(&bars.v_full[s]); };
  auto b_e = [&](int s) { return smem_u32(&bars.kv_empty[s]); };
  auto b_s = [&](int h) { return smem_u32(&bars.s_full[h]); };
  auto b_f = [&](int h) { return smem_u32(&bars.s_free[h]); };
  auto b_p = [&](int h) { return smem_u32(&bars.p_full[h]); };
  auto b_o = [&](int h) { return smem_u32(&bars.o_done[h]); };
  auto b_of = [&](int h) { return smem_u32(&bars.o_free[h]); };
  auto b_osq = [&](int h) { return smem_u32(&bars.ostage_full[h]); };
  auto b_osf = [&](int h) { return smem_u32(&bars.ostage_free[h]); };

  if (threadIdx.x == 0) {
    for (int r = 0; r < kRing; ++r) {
      mbar_init(b_if(r), 1);
      mbar_init(b_ie(r), NH * 128 + C::MW);  // every softmax thread and each MMA warp
    }
    for (int b = 0; b < C::QBUF; ++b) {
      mbar_init(b_qf(b), 1);
      mbar_init(b_qe(b), C::MW);
    }
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(b_k(s), 1);
      mbar_init(b_v(s), 1);
      mbar_init(b_e(s), C::MW);  // one commit per MMA warp
    }
    for (int h = 0; h < NH; ++h) {
      mbar_init(b_s(h), 1);
      mbar_init(b_f(h), 128);
      mbar_init(b_p(h), 128);
      mbar_init(b_o(h), 1);
      mbar_init(b_of(h), 128);
      mbar_init(b_osq(h), 128);
      mbar_init(b_osf(h), 1);
      for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&bars.turn[h][q]), 1);
    }
    mbar_init(smem_u32(&bars.never), 1);
    bars.abort = 0;
    mbar_fence_init();
  }
  if (warp == C::MMA_WARP) tmem_alloc(smem_u32(&bars.tmem), C::TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = bars.tmem;
  volatile int32_t(*ring)[8] = bars.ring;
  // the item the producer decoded into ring slot `slot` (w >= n_items ends the list)
  auto ring_item = [&](int slot, int &w, Item &it, int &e0) {
    w = ring[slot][0];
    it.qt.row0 = ring[slot][1];
    it.qt.row1 = ring[slot][2];
    it.qt.ent0 = ring[slot][3];
    it.qt.ent1 = ring[slot][4];
    it.h0 = ring[slot][5];
    it.g = ring[slot][6];
    e0 = ring[slot][7];
    it.n = it.qt.ent1 - it.qt.ent0;
  };

  if (warp >= 4 * NH) {
    if (C::SPLIT) regs_dec<C::SERVICE_REGS>();
    if (warp == C::PROD_WARP) {
      // ---------------------------------------------------------- producer (whole warp, one lane issues)
      if (elect_one()) {
        prefetch_map(&mq);
        prefetch_map(&mk);
        prefetch_map(&mv);
        if (G) {
          prefetch_map(&mkg);
          prefetch_map(&mvg);
        }
      }
      __syncwarp();
      // Q, K, V may come from the kernel before this one in the stream (RoPE):
      // everything above overlapped its tail; every read of them starts here
      griddep_wait();
      int t = 0, j = 0, fetched = 0;
      bool ok = true;
      if (a.self_test) {
        // timeout self-test: before any copy or MMA is issued, wait 2 ms on a
        // barrier nothing arrives on; the wait gives up, writes TREE_ERR_TIMEOUT
        // and raises the CTA's abort flag, and every role winds down
        ok = wait_bar(smem_u32(&bars.never), 0, abort, a.status, true, kSelfTestNs);
        ok = __all_sync(0xffffffffu, ok);
      }
      // the Q tile(s) of item `qi` into buffer qb
      auto issue_q = [&](int qb, const Item &qi) {
        if (elect_one()) {
          mbar_expect_tx(b_qf(qb), C::Q_BYTES);
#pragma unroll
          for (int h = 0; h < NH; ++h)
#pragma unroll
            for (int c = 0; c < C::CB; ++c) {
              const uint32_t dst = s_base + C::Q_OFF + qb * C::Q_BYTES + (h * C::CB + c) * BOX_BYTES;
              if (HP) {
                // tpm rows of each q head, one box each (tpm >= 16: every sub-box starts on a
                // 1024-byte swizzle period, so the tile is laid out as one 128-row box)
                for (int hh = 0; hh < a.ratio; ++hh)
                  tma_load_2d(dst + hh * a.tpm * 128, &mq, (qi.h0 + hh) * D + 64 * c,
                              qi.qt.row0 - a.q0 + h * a.tpm, b_qf(qb));
              } else {
                tma_load_2d(dst, &mq, (qi.h0 + h) * D + 64 * c, qi.qt.row0 - a.q0, b_qf(qb));
              }
            }
        }
        __syncwarp();
      };
      while (ok) {
        // claim the next item and publish it in the ring (a value >= n_items ends the list)
        const int slot = fetched % kRing;
        if (fetched >= kRing && !(ok = wait_bar_warp(b_ie(slot), ((fetched / kRing) - 1) & 1, abort, a.status)))
          break;
        int w = 0;
        if (lane == 0) w = a.work ? atomicAdd(a.work, 1) : (int)blockIdx.x + fetched * (int)gridDim.x;
        w = __shfl_sync(0xffffffffu, w, 0);
        ++fetched;
        // decoded here, so that the consumers read the item from shared memory
        Item it{};
        int e0 = 0;
        if (w < a.n_items) {
          it = item_at<NH, HP>(a, w);
          if (it.n > 0) e0 = __ldg(a.ent + it.qt.ent0);
        }
        if (lane == 0) {
          ring[slot][0] = w;
          ring[slot][1] = it.qt.row0;
          ring[slot][2] = it.qt.row1;
          ring[slot][3] = it.qt.ent0;
          ring[slot][4] = it.qt.ent1;
          ring[slot][5] = it.h0;
          ring[slot][6] = it.g;
          ring[slot][7] = e0;
          mbar_arrive(b_if(slot));
        }
        __syncwarp();
        if (w >= a.n_items) {
          // no more items for this CTA: the next kernel in the stream may start launching
          griddep_launch();
          break;
        }
        if (it.n <= 0) continue;  // (a plan never makes one: every query tile sees its own rows)
        const int b = j % C::QBUF;
        if (j >= C::QBUF && !(ok = wait_bar_warp(b_qe(b), ((j / C::QBUF) - 1) & 1, abort, a.status))) break;
        issue_q(b, it);
        for (int i = 0; i < it.n; ++i, ++t) {
          const int st = t % C::STAGES;
          if (t >= C::STAGES && !(ok = wait_bar_warp(b_e(st), ((t / C::STAGES) - 1) & 1, abort, a.status))) break;
          if (G) {
            // tiling by position: a contiguous entry is one tiled box like a packed key
            // tile; otherwise its 128 keys are gathered row by row (lane l loads slots
            // 4l .. 4l + 3).  Its run table comes with the keys.
            const int ev = __ldg(a.ent + it.qt.ent0 + i);
            if ((ev & 3) == 2) {
              // a full contiguous range: one tiled box of keys from (ev >> 2), no run table
              if (elect_one()) {
                const uint32_t vb = C::KV_ONE ? b_k(st) : b_v(st);
                mbar_expect_tx(b_k(st), (C::KV_ONE ? 2 : 1) * C::CB * BOX_BYTES);
#pragma unroll
                for (int c = 0; c < C::CB; ++c)
                  tma_load_2d(s_base + C::K_OFF + (st * C::CB + c) * BOX_BYTES, &mk, it.g * D + 64 * c, ev >> 2, b_k(st));
                if (!C::KV_ONE) mbar_expect_tx(vb, C::CB * BOX_BYTES);
#pragma unroll
                for (int c = 0; c < C::CB; ++c)
                  tma_load_2d(s_base + C::V_OFF + (st * C::CB + c) * BOX_BYTES, &mv, it.g * D + 64 * c, ev >> 2, vb);
              }
              __syncwarp();
              continue;
            }
            const int e = ev >> 2;
            if (a.boxes && !(ev & 2)) {
              // gathered tile (tiling 2): lane r loads the slots of run r, widened to whole
              // groups of 8 rows, as tiled boxes of 8, 16, 32, 64 or 128 rows.  A stretch of
              // consecutive keys starts at a multiple of 8 slots, so every box lands on a
              // 1024-byte swizzle period; where two runs of one stretch share a group of 8 both
              // write the same keys there, and rows past a stretch (keys of other blocks, or the
              // fill value past the last key) go to slots no run covers.
              const int32_t *vr = a.vruns + (size_t)e * kVRunWords;
              const int R = __ldg(vr);
              int4 run = make_int4(0, -1, 0, 0);
              if (lane < R) run = __ldg(reinterpret_cast<const int4 *>(vr + 8) + lane);
              // the last run loads through slot 127: every slot then holds finite keys and
              // values (an unloaded V row could hold NaN, and 0 * NaN would reach O)
              const int s0 = run.x & ~7;
              const int nr = lane < R ? (lane == R - 1 ? 127 : (run.y | 7)) - s0 + 1 : 0;
              const uint32_t kb = __reduce_add_sync(0xffffffffu, (uint32_t)nr) * 128u * C::CB;
              const uint32_t v_bar = C::KV_ONE ? b_k(st) : b_v(st);
              if (lane == 0) {
                mbar_expect_tx(b_k(st), (C::KV_ONE ? 2 : 1) * kb + kVRunWords * 4);
                bulk_load(s_base + C::RUNS_OFF + st * 512, vr, kVRunWords * 4, b_k(st));
                if (!C::KV_ONE) mbar_expect_tx(v_bar, kb);
              }
              __syncwarp();
              if (nr > 0) {
                int y = run.z - (run.x - s0), slot = s0;
#pragma unroll
                for (int lg = 4; lg >= 0; --lg) {  // boxes of 8 << lg rows
                  if (!(((nr >> 3) >> lg) & 1)) continue;
                  const CUtensorMap *km = lg == 4 ? &mk : &bm.k[lg], *vm = lg == 4 ? &mv : &bm.v[lg];
#pragma unroll
                  for (int c = 0; c < C::CB; ++c)
                    tma_load_2d(s_base + C::K_OFF + (st * C::CB + c) * BOX_BYTES + slot * 128, km, it.g * D + 64 * c,
                                y, b_k(st));
#pragma unroll
                  for (int c = 0; c < C::CB; ++c)
                    tma_load_2d(s_base + C::V_OFF + (st * C::CB + c) * BOX_BYTES + slot * 128, vm, it.g * D + 64 * c,
                                y, v_bar);
                  slot += 8 << lg;
                  y += 8 << lg;
                }
              }
              __syncwarp();
              continue;
            }
            const int4 rows = __ldg(reinterpret_cast<const int4 *>(a.vkeys + (size_t)e * BN) + lane);
            const int jc = __shfl_sync(0xffffffffu, rows.x, 0);  // slot 0's key
            const uint32_t v_bar = C::KV_ONE ? b_k(st) : b_v(st);
            if (lane == 0) {
              mbar_expect_tx(b_k(st), (C::KV_ONE ? 2 : 1) * C::CB * BOX_BYTES + kVRunWords * 4);
              bulk_load(s_base + C::RUNS_OFF + st * 512, a.vruns + (size_t)e * kVRunWords, kVRunWords * 4, b_k(st));
              if (!C::KV_ONE) mbar_expect_tx(v_bar, C::CB * BOX_BYTES);
            }
            __syncwarp();
            if (ev & 2) {
              if (lane == 0) {
#pragma unroll
                for (int c = 0; c < C::CB; ++c)
                  tma_load_2d(s_base + C::K_OFF + (st * C::CB + c) * BOX_BYTES, &mk, it.g * D + 64 * c, jc, b_k(st));
#pragma unroll
                for (int c = 0; c < C::CB; ++c)
                  tma_load_2d(s_base + C::V_OFF + (st * C::CB + c) * BOX_BYTES, &mv, it.g * D + 64 * c, jc, v_bar);
              }
            } else {
              // Lanes 2g and 2g+1 hold the 8 slots of group g.  A group whose slots hold
              // consecutive keys, or no key at all (slot keys 0), loads as one tiled box of 8
              // rows (from its first key, or rows 0-7) that lands on its 1024-byte swizzle
              // period; only the groups where block pieces meet are gathered row by row.
              const bool c4 = rows.y == rows.x + 1 && rows.z == rows.x + 2 && rows.w == rows.x + 3;
              const bool z4 = (rows.x | rows.y | rows.z | rows.w) == 0;
              const int nb_first = __shfl_xor_sync(0xffffffffu, rows.x, 1);
              const bool nb_c4 = __shfl_xor_sync(0xffffffffu, c4, 1), nb_z4 = __shfl_xor_sync(0xffffffffu, z4, 1);
              const bool g_box = (z4 && nb_z4) ||
                                 (c4 && nb_c4 && ((lane & 1) ? rows.x == nb_first + 4 : nb_first == rows.x + 4));
              if (g_box) {
                if (!(lane & 1)) {
#pragma unroll
                  for (int c = 0; c < C::CB; ++c)
                    tma_load_2d(s_base + C::K_OFF + (st * C::CB + c) * BOX_BYTES + lane * 512, &bm.k[0],
                                it.g * D + 64 * c, rows.x, b_k(st));
#pragma unroll
                  for (int c = 0; c < C::CB; ++c)
                    tma_load_2d(s_base + C::V_OFF + (st * C::CB + c) * BOX_BYTES + lane * 512, &bm.v[0],
                                it.g * D + 64 * c, rows.x, v_bar);
                }
              } else {
#pragma unroll
                for (int c = 0; c < C::CB; ++c)
                  tma_gather4(s_base + C::K_OFF + (st * C::CB + c) * BOX_BYTES + lane * 512, &mkg, it.g * D + 64 * c,
                              rows, b_k(st));
#pragma unroll
                for (int c = 0; c < C::CB; ++c)
                  tma_gather4(s_base + C::V_OFF + (st * C::CB + c) * BOX_BYTES + lane * 512, &mvg, it.g * D + 64 * c,
                              rows, v_bar);
              }
            }
            __syncwarp();
            continue;
          }
          const int j0 = (__ldg(a.ent + it.qt.ent0 + i) >> 1) * BN;
          if (elect_one()) {
            // with three stages K, the keys' subtree ends and V complete one
            // barrier (the loads run far enough ahead that V is in place before
            // the QK is issued); with two, V has its own
            const uint32_t v_bar = C::KV_ONE ? b_k(st) : b_v(st);
            mbar_expect_tx(b_k(st), (C::KV_ONE ? 2 : 1) * C::CB * BOX_BYTES + kRunWords * 4);
#pragma unroll
            for (int c = 0; c < C::CB; ++c)
              tma_load_2d(s_base + C::K_OFF + (st * C::CB + c) * BOX_BYTES, &mk, it.g * D + 64 * c, j0, b_k(st));
            bulk_load(s_base + C::RUNS_OFF + st * 512, a.runs + (size_t)(j0 / BN) * kRunWords, kRunWords * 4, b_k(st));
            if (!C::KV_ONE) mbar_expect_tx(v_bar, C::CB * BOX_BYTES);
#pragma unroll
            for (int c = 0; c < C::CB; ++c)
              tma_load_2d(s_base + C::V_OFF + (st * C::CB + c) * BOX_BYTES, &mv, it.g * D + 64 * c, j0, v_bar);
          }
          __syncwarp();
        }
        ++j;
      }
      // wind down: every copy issued must have landed before the CTA exits
      for (int u = (t > C::STAGES ? t - C::STAGES : 0); u < t; ++u) {
        wait_bar(b_k(u % C::STAGES), (u / C::STAGES) & 1, abort, nullptr, false, kDrainNs);
        if (!C::KV_ONE) wait_bar(b_v(u % C::STAGES), (u / C::STAGES) & 1, abort, nullptr, false, kDrainNs);
      }
      for (int u = (j > C::QBUF ? j - C::QBUF : 0); u < j; ++u)
        wait_bar(b_qf(u % C::QBUF), (u / C::QBUF) & 1, abort, nullptr, false, kDrainNs);
    } else if (warp >= C::MMA_WARP && warp < C::MMA_WARP + C::MW) {
      // ---------------------------------------------------------- MMA issuer of q heads h0 + [hb, he)
      // One lane issues.  At d = 64 each head has its own MMA warp, so that the
      // heads' chains of waits run on their own and their MMAs interleave on
      // the tensor core as operands become ready; at d = 128 (P over S) one
      // warp orders both heads, PV_h then the next QK_h, head after head.
      const int hb = (warp - C::MMA_WARP) * (NH / C::MW), he = hb + NH / C::MW;
      constexpr uint32_t idesc_qk = idesc_f16(128, 128, false);
      constexpr uint32_t idesc_pv = idesc_f16(128, D, true);
      // Descriptors are built once per operand tile and advanced by constant
      // offsets (the start-address field holds address / 16 in its low bits).
      const uint64_t q_desc0 = sdesc_sw128(s_base + C::Q_OFF, 16, 1024);
      const uint64_t k_desc0 = sdesc_sw128(s_base + C::K_OFF, 16, 1024);
      const uint64_t v_desc0 = sdesc_sw128(s_base + C::V_OFF, BOX_BYTES, 1024);
      auto issue_qk = [&](int h, int qb, int st) {
        const uint64_t da0 = q_desc0 + ((qb * C::Q_BYTES + h * C::CB * BOX_BYTES) >> 4);
        const uint64_t db0 = k_desc0 + ((st * C::CB * BOX_BYTES) >> 4);
        const uint32_t s_tmem = tmem + 128 * h;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * BOX_BYTES + (kk & 3) * 32) >> 4;
            mma_ss(s_tmem, da0 + off, db0 + off, idesc_qk, kk > 0);
          }
          mma_commit(b_s(h));
        }
        __syncwarp();
      };
      auto issue_pv = [&](int h, int st, bool accumulate) {
        const uint32_t p_tmem = tmem + (C::PSEP ? C::P_COL + 64 * h : 128 * h);
        const uint32_t o_tmem = tmem + C::O_COL + D * h;
        const uint64_t db0 = v_desc0 + ((st * C::CB * BOX_BYTES) >> 4);
        const uint32_t acc0 = accumulate ? 1u : 0u;
        if (elect_one()) {
          mma_ts(o_tmem, p_tmem, db0, idesc_pv, acc0);
#pragma unroll
          for (int kk = 1; kk < BN / 16; ++kk) mma_ts(o_tmem, p_tmem + 8 * kk, db0 + kk * (2048 >> 4), idesc_pv, 1u);
          mma_commit(b_o(h));
        }
        __syncwarp();
      };
      auto commit = [&](uint32_t bar) {
        if (elect_one()) mma_commit(bar);
        __syncwarp();
      };
      // items from the ring, in order; skips items without key tiles
      int taken = 0;
      auto next_item = [&](Item &out) -> int {  // 1: item, 0: list ended, -1: gave up
        for (;;) {
          const int slot = taken % kRing;
          if (!wait_bar_warp(b_if(slot), (taken / kRing) & 1, abort, a.status)) return -1;
          int w, e0;
          ring_item(slot, w, out, e0);
          __syncwarp();
          if (elect_one()) mbar_arrive(b_ie(slot));
          __syncwarp();
          ++taken;
          if (w >= a.n_items) return 0;
          if (out.n > 0) return 1;
        }
      };
      Item cur;
      int got = next_item(cur);
      bool ok = got >= 0;
      int jc = 0, ic = 0, T = 0, last_qk = -1;
      // prologue: S of the first tile
      if (got == 1) {
        ok = wait_bar_warp(b_qf(0), 0, abort, a.status) && wait_bar_warp(b_k(0), 0, abort, a.status);
        if (ok) {
          fence_after();
          for (int h = hb; h < he; ++h) issue_qk(h, 0, 0);
          last_qk = 0;
          if (cur.n == 1) commit(b_qe(0));
        }
      }
      while (ok && got == 1) {
        // the tile after T: the next tile of this item, or the first of the next item
        int jn = jc, in = ic + 1;
        Item nxt = cur;
        bool has_next = in < cur.n;
        if (!has_next) {
          const int g2 = next_item(nxt);
          if (g2 < 0) {
            ok = false;
            break;
          }
          has_next = g2 == 1;
          in = 0;
          jn = jc + 1;
        }
        const int qbn = jn % C::QBUF, stn = (T + 1) % C::STAGES;
        // operands of the next S: its Q tile (first tile of an item) and its K tile
        auto wait_next_operands = [&]() {
          if (in == 0 && !wait_bar_warp(b_qf(qbn), (jn / C::QBUF) & 1, abort, a.status)) return false;
          return wait_bar_warp(b_k(stn), ((T + 1) / C::STAGES) & 1, abort, a.status);
        };
        if (C::PSEP && has_next) {
          // next S first: S_h is free once the softmax has read it into registers
          if (!(ok = wait_next_operands())) break;
          for (int h = hb; h < he && ok; ++h) {
            if (!(ok = wait_bar_warp(b_f(h), T & 1, abort, a.status))) break;
            fence_after();
            issue_qk(h, qbn, stn);
            last_qk = T + 1;
          }
          if (!ok) break;
          if (in == nxt.n - 1) commit(b_qe(qbn));  // the Q buffer is free once these QKs have read it
        }
        const int st = T % C::STAGES;
        if (!C::KV_ONE && !(ok = wait_bar_warp(b_v(st), (T / C::STAGES) & 1, abort, a.status))) break;
        for (int h = hb; h < he && ok; ++h) {
          if (!(ok = wait_bar_warp(b_p(h), T & 1, abort, a.status))) break;
          // a new item's first PV overwrites O_h: its previous values must have been read
          if (ic == 0 && jc > 0 && !(ok = wait_bar_warp(b_of(h), (jc - 1) & 1, abort, a.status))) break;
          fence_after();
          issue_pv(h, st, ic > 0);
          if (!C::PSEP && has_next) {
            // P_h shares S_h's columns: the next S_h waits until this PV has read P_h
            if (h == hb && !(ok = wait_next_operands())) break;
            if (!(ok = wait_bar_warp(b_o(h), T & 1, abort, a.status))) break;
            fence_after();
            issue_qk(h, qbn, stn);
            last_qk = T + 1;
          }
        }
        if (!ok) break;
        if (!C::PSEP && has_next && in == nxt.n - 1) commit(b_qe(qbn));
        commit(b_e(st));
        ++T;
        if (!has_next) break;
        jc = jn;
        ic = in;
        cur = nxt;
      }
      // wind down: every MMA this warp issued (and the commits after it) has
      // completed, and every stage's release has landed, before the CTA exits
      if (T > 0) {
        for (int h = hb; h < he; ++h) wait_bar(b_o(h), (T - 1) & 1, abort, nullptr, false, kDrainNs);
        for (int u = (T > C::STAGES ? T - C::STAGES : 0); u < T; ++u)
          wait_bar(b_e(u % C::STAGES), (u / C::STAGES) & 1, abort, nullptr, false, kDrainNs);
      }
      if (!ok && last_qk >= 0)
        for (int h = hb; h < he; ++h) wait_bar(b_s(h), last_qk & 1, abort, nullptr, false, kDrainNs);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    if (C::SPLIT) regs_inc<C::SOFTMAX_REGS>();
    const int h = warp >> 2;
    const int r = 32 * (warp & 3) + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t tS = t_lane + 128 * h;
    const uint32_t tP = C::PSEP ? t_lane + C::P_COL + 64 * h : tS;
    const uint32_t tO = t_lane + C::O_COL + D * h;
    bool ok = true;
    int T = 0, stage_uses = 0;
    // With DEFER the epilogue of an item waits until the P of the next item's
    // first tile is stored: the wait for the item's last PV then overlaps that
    // tile's arithmetic.  The finished item's state waits here meanwhile.
    bool pend = false;
    Item pit{};
    int piq = 0;
    float pm = 0.f, pl = 0.f;
    auto epilogue = [&]() -> bool {
      // ---- read O_h, hand its columns back, then O / l -> f16 rows
      if (!wait_bar_warp(b_o(h), (T - 1) & 1, abort, a.status)) return false;
      fence_after();
      uint32_t o[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + 32 * c, o + 32 * c);
      tmem_wait_ld();
      fence_before();
      mbar_arrive(b_of(h));
      // O / l as f16 into this head's 128-byte-swizzled staging box, 64 columns at
      // a time; row 0's thread issues one TMA store per box once every row is
      // written.  It waits for a store to have read the box only when the box
      // is next needed (normally an item later, long done), and then hands it
      // back, so no warp stalls on the store here.  Rows past the chunk are
      // clipped by the store.
      const float inv = 1.f / pl;
      const uint32_t stage = s_base + C::O_OFF + h * BOX_BYTES;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int use = stage_uses++;
        if (use > 0) {
          if (r == 0) {
            bulk_wait_read0();
            mbar_arrive(b_osf(h));
          }
          if (!wait_bar_warp(b_osf(h), (use - 1) & 1, abort, a.status)) return false;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t *x = o + 64 * c + 8 * u;
          const uint4 v4 = make_uint4(pack_f16x2(__uint_as_float(x[0]) * inv, __uint_as_float(x[1]) * inv),
                                      pack_f16x2(__uint_as_float(x[2]) * inv, __uint_as_float(x[3]) * inv),
                                      pack_f16x2(__uint_as_float(x[4]) * inv, __uint_as_float(x[5]) * inv),
                                      pack_f16x2(__uint_as_float(x[6]) * inv, __uint_as_float(x[7]) * inv));
          const uint32_t addr = stage + r * 128 + ((u ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v4.x), "r"(v4.y), "r"(v4.z),
                       "r"(v4.w)
                       : "memory");
        }
        fence_async_shared();
        mbar_arrive(b_osq(h));
        if (r == 0 && wait_bar(b_osq(h), use & 1, abort, a.status)) {
          if (HP) {
            // rows past the query tile are clipped by the store (they lie past the chunk);
            // a half that starts past it stores nothing
            if (pit.qt.row0 + h * a.tpm < pit.qt.row1)
              for (int hh = 0; hh < a.ratio; ++hh)
                tma_store_2d(&mo, (pit.h0 + hh) * D + 64 * c, pit.qt.row0 - a.q0 + h * a.tpm,
                             stage + hh * a.tpm * 128);
          } else {
            tma_store_2d(&mo, (pit.h0 + h) * D + 64 * c, pit.qt.row0 - a.q0, stage);
          }
          bulk_commit();
        }
      }
      if (a.lse && piq < pit.qt.row1) {
        const float mu = (pm == -INFINITY) ? 0.f : pm;
        a.lse[(size_t)(piq - a.q0) * a.hq + pit.h0 + (HP ? r / a.tpm : h)] = (mu + __log2f(pl)) * 0.69314718055994531f;
      }
      pend = false;
      return true;
    };
    for (int taken = 0; ok; ++taken) {
      const int slot = taken % kRing;
      if (!(ok = wait_bar_warp(b_if(slot), (taken / kRing) & 1, abort, a.status))) break;
      int w, e_next;
      Item it;
      ring_item(slot, w, it, e_next);
      mbar_arrive(b_ie(slot));
      if (w >= a.n_items) break;
      if (it.n <= 0) continue;
      // this thread's row of the query tile: its token, and (packed heads) its q head's rows
      const int srow = HP ? h * a.tpm + (r & (a.tpm - 1)) : r;
      const int iq = it.qt.row0 + srow;
      float m = -INFINITY, l = 0.f;
      for (int i = 0; i < it.n; ++i, ++T) {
        const int st = T % C::STAGES;
        const int e = e_next;  // the next tile's entry loads while this one is processed
        if (i + 1 < it.n) e_next = __ldg(a.ent + it.qt.ent0 + i + 1);
        // a partial tile also needs the run table of its keys (same stage as K)
        if ((e & 1) && !(ok = wait_bar_warp(b_k(st), (T / C::STAGES) & 1, abort, a.status))) break;
        if (!(ok = wait_bar_warp(b_s(h), T & 1, abort, a.status))) break;
        fence_after();
        uint32_t s[128];
        tmem_ld32(tS + 0, s);
        tmem_ld32(tS + 32, s + 32);
        tmem_ld32(tS + 64, s + 64);
        tmem_ld32(tS + 96, s + 96);
        tmem_wait_ld();
        if (C::PSEP) {
          fence_before();
          mbar_arrive(b_f(h));  // S_h may be overwritten by the next QK
        }
        const uint32_t my_turn = smem_u32(&bars.turn[h][warp & 3]), other_turn = smem_u32(&bars.turn[h ^ 1][warp & 3]);
        if (C::ALT) {
          // head 1 computes tile T after head 0 has; head 0 computes tile T after head 1 has computed T - 1
          if (h == 1 && !(ok = wait_bar_warp(other_turn, T & 1, abort, a.status))) break;
          if (h == 0 && T > 0 && !(ok = wait_bar_warp(other_turn, (T - 1) & 1, abort, a.status))) break;
        }
        if (G && (e & 1)) {
          // tiling by position: rows not assigned to this entry take nothing from it;
          // an assigned row sees slot c of run r iff c - c0 <= iq - j0 and j0 <= iq < send
          const int32_t *tb = sRuns + st * 128;
          uint32_t mw[4] = {0u, 0u, 0u, 0u};
          if ((tb[4 + (srow >> 5)] >> (srow & 31)) & 1) {
            const int R = tb[0];
#pragma unroll
            for (int rr = 0; rr < kMaxRuns; ++rr) {
              if (rr >= R) break;
              const int4 run = reinterpret_cast<const int4 *>(tb + 8)[rr];  // c0, c1, j0, send
              if (iq >= run.z && iq < run.w) {
                const int lo = run.x, hi = min(run.y, run.x + (iq - run.z));
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  const int a0 = max(lo, 32 * q4) - 32 * q4, a1 = min(hi, 32 * q4 + 31) - 32 * q4;
                  if (a0 <= a1) mw[q4] |= (0xffffffffu >> (31 - (a1 - a0))) << a0;
                }
              }
            }
          }
#pragma unroll
          for (int c = 0; c < 128; ++c)
            s[c] = (mw[c >> 5] & (1u << (c & 31))) ? s[c] : __float_as_uint(-INFINITY);
        } else if (e & 1) {
          // partial tile: key j = j0 + c is visible iff j <= iq < send[j].  The
          // row's 128-bit mask (the runs of the tile that end after the query,
          // cut at the query's own column), then one bit test per score.
          const int j0 = (e >> 1) * BN;
          const int cmax = iq - j0;  // keys c <= cmax are not after the query
          const int32_t *tb = sRuns + st * 128;
          const int R = tb[0];
          uint32_t mw0 = 0u, mw1 = 0u, mw2 = 0u, mw3 = 0u;
          if (R <= kMaxRuns) {
#pragma unroll
            for (int rr = 0; rr < kMaxRuns; ++rr) {
              if (rr >= R) break;
              const bool vis = iq < tb[4 + rr];
              const uint4 b = reinterpret_cast<const uint4 *>(tb + 20)[rr];
              mw0 |= vis ? b.x : 0u;
              mw1 |= vis ? b.y : 0u;
              mw2 |= vis ? b.z : 0u;
              mw3 |= vis ? b.w : 0u;
            }
          } else {
            // many short blocks: test the keys' subtree ends one by one
            const int4 *sd = reinterpret_cast<const int4 *>(a.send + j0);
#pragma unroll 1
            for (int c4 = 0; c4 < 32; ++c4) {
              const int4 se = __ldg(sd + c4);
              const uint32_t nib = (uint32_t)(iq < se.x) | ((uint32_t)(iq < se.y) << 1) |
                                   ((uint32_t)(iq < se.z) << 2) | ((uint32_t)(iq < se.w) << 3);
              const uint32_t bit = nib << (4 * (c4 & 7));
              const int q = c4 >> 3;
              mw0 |= q == 0 ? bit : 0u;
              mw1 |= q == 1 ? bit : 0u;
              mw2 |= q == 2 ? bit : 0u;
              mw3 |= q == 3 ? bit : 0u;
            }
          }
          uint32_t mw[4] = {mw0, mw1, mw2, mw3};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int k = cmax - 32 * q4;
            mw[q4] &= k >= 31 ? 0xffffffffu : (k < 0 ? 0u : (0xffffffffu >> (31 - k)));
          }
#pragma unroll
          for (int c = 0; c < 128; ++c)
            s[c] = (mw[c >> 5] & (1u << (c & 31))) ? s[c] : __float_as_uint(-INFINITY);
        }
        // row maximum: three-input max over four independent chains
        float mx4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) mx4[u] = __uint_as_float(s[u]);
#pragma unroll
        for (int c = 4; c < 128; c += 8)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            mx4[u] = max3(mx4[u], __uint_as_float(s[c + 2 * u]), __uint_as_float(s[c + 2 * u + 1]));
        const float mx = max3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
        const float mt = mx * a.scale_log2;  // -inf stays -inf (scale > 0)
        const bool grow = mt > m + 8.f;      // also true for the first finite maximum
        float alpha = 1.f;
        if (grow) {
          alpha = ex2(m - mt);  // 0 when m is -inf
          m = mt;
        }
        const float mu = (m == -INFINITY) ? 0.f : m;
        // p = 2^(s * scale_log2 - mu) on pairs of lanes (paired fma and add)
        const uint64_t scale2 = f32x2(a.scale_log2, a.scale_log2), nmu2 = f32x2(-mu, -mu);
        uint64_t sum2[4] = {0, 0, 0, 0};
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          float x0, x1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), scale2, nmu2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          sum2[(c >> 1) & 3] = add_f32x2(sum2[(c >> 1) & 3], f32x2(p0, p1));
          s[c >> 1] = pack_f16x2(p0, p1);
        }
        float sl[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) f32x2_split(sum2[u], sl[2 * u], sl[2 * u + 1]);
        l = l * alpha + (((sl[0] + sl[1]) + (sl[2] + sl[3])) + ((sl[4] + sl[5]) + (sl[6] + sl[7])));
        if (C::ALT) {
          __syncwarp();
          if (lane == 0) mbar_arrive(my_turn);
        }
        // PV_h of the previous tile must be done before P_h is rewritten
        // (separate P) or O_h is rescaled
        const bool need_o = i > 0 && __any_sync(0xffffffffu, grow);
        if ((i > 0 || pend) && (C::PSEP || need_o)) {
          if (!(ok = wait_bar_warp(b_o(h), (T - 1) & 1, abort, a.status))) break;
          fence_after();
        }
        tmem_st32(tP + 0, s);
        tmem_st32(tP + 32, s + 32);
        if (need_o) {
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
            tmem_st32(tO + 32 * c, o);
          }
        }
        tmem_wait_st();
        fence_before();
        mbar_arrive(b_p(h));
        // the previous item's epilogue, now that this item's first P is stored
        // (its first PV waits for the previous O to be read)
        if (pend && !(ok = epilogue())) break;
      }
      if (!ok) break;
      pend = true;
      pit = it;
      piq = iq;
      pm = m;
      pl = l;
      if (!C::DEFER && !(ok = epilogue())) break;
    }
    if (ok && pend) ok = epilogue();
    if (r == 0) bulk_wait0();  // every output store has completed
  }
  fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (a.work && threadIdx.x == 0) {
    // the last CTA to finish (all claims are done by then) resets the counter
    __threadfence();
    if (atomicAdd(a.work + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(a.work, 0);
      atomicExch(a.work + 1, 0);
    }
  }
}

template <int D, int NH>
int launch_tc(const Plan &P, const int32_t *img, int chunk, const void *q, const void *k, const void *v, void *o,
              float *lse, int hq, int hkv, float scale, int32_t *work, int32_t self_test, int32_t *status,
              cudaStream_t s) {
  using C = Cfg<D, NH>;
  const bool gather = P.tiling != 0;
  // packed heads (NH == 2 only): tokens per MMA tile, the Q and O boxes' height
  const bool hp = NH == 2 && P.pack_heads > 1;
  const int tpm = hp ? BN / P.pack_heads : BN;
  auto kern = gather ? tree_attn_tc<D, NH, true, false> : tree_attn_tc<D, NH, false, false>;
  if constexpr (NH == 2)
    if (hp) kern = tree_attn_tc<D, NH, true, true>;
  int rc = set_max_dynamic_smem(reinterpret_cast<const void *>(kern), (int)C::SMEM, "tree_attn_fwd");
  if (rc) return rc;
  const int32_t q0 = P.chunk_q0[chunk], nq = P.chunk_q1[chunk] - q0;
  CUtensorMap mq, mk, mv, mo, mkg, mvg;
  BoxMaps bm;
  std::memset(&bm, 0, sizeof bm);
  if ((rc = make_map(&mq, q, (int64_t)hq * D, nq, "tree_attn_fwd", tpm)) ||
      (rc = make_map(&mk, k, (int64_t)hkv * D, P.n_tot, "tree_attn_fwd")) ||
      (rc = make_map(&mv, v, (int64_t)hkv * D, P.n_tot, "tree_attn_fwd")) ||
      (rc = make_map(&mkg, k, (int64_t)hkv * D, P.n_tot, "tree_attn_fwd", 1)) ||
      (rc = make_map(&mvg, v, (int64_t)hkv * D, P.n_tot, "tree_attn_fwd", 1)) ||
      (rc = make_map(&mo, o, (int64_t)hq * D, nq, "tree_attn_fwd", tpm)))
    return rc;
  if (P.tiling != 0)
    for (int lg = 0; lg < 4; ++lg)
      if ((rc = make_map(&bm.k[lg], k, (int64_t)hkv * D, P.n_tot, "tree_attn_fwd", 8 << lg)) ||
          (rc = make_map(&bm.v[lg], v, (int64_t)hkv * D, P.n_tot, "tree_attn_fwd", 8 << lg)))
        return rc;
  AttnArgs a;
  a.send = img + P.off_send;
  a.runs = img + P.off_runs;
  a.vkeys = img + P.off_vkeys;
  a.vruns = img + P.off_vruns;
  a.qtiles = reinterpret_cast<const QTile *>(img + P.off_qtile);
  a.ent = img + P.off_ent;
  a.order = img + P.off_order;
  a.o = reinterpret_cast<__half *>(o);
  a.lse = lse;
  a.status = status;
  a.t0 = P.chunk_t0[chunk];
  a.q0 = q0;
  a.n_tot = P.n_tot;
  a.hq = hq;
  a.hkv = hkv;
  a.ratio = hq / hkv;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.self_test = self_test;
  const int tiles = P.chunk_t1[chunk] - P.chunk_t0[chunk];
  a.tpm = tpm;
  a.boxes = P.tiling == 2;
  a.n_items = tiles * hkv * (hp ? 1 : a.ratio / NH);
  a.work = work;
  if (a.n_items == 0) return TREE_OK;
  const dim3 grid((unsigned)std::min(a.n_items, sm_count()));
  const cudaError_t e = launch_dependent(kern, grid, dim3(C::THREADS), C::SMEM, s, mq, mk, mv, mo, mkg, mvg, bm, a);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_attn_fwd: launch failed: %s", cudaGetErrorString(e));
  return launch_status("tree_attn_fwd");
}

}  // namespace
}  // namespace tree

extern "C" TREE_API int tree_attn_fwd(const tree_plan_t *plan, const void *plan_dev, int32_t chunk,
                                      const void *q, const void *k, const void *v, void *o, float *lse,
                                      const tree_attn_params_t *params, int32_t *status, tree_stream_t stream) {
  using namespace tree;
  if (!plan || !plan_dev || !q || !k || !v || !o || !params)
    return fail(TREE_ERR_INVALID_ARG, "tree_attn_fwd: NULL argument");
  const Plan &P = plan->p;
  if (chunk < 0 || chunk >= P.n_chunks)
    return fail(TREE_ERR_INVALID_ARG, "tree_attn_fwd: chunk %d out of range [0, %d)", chunk, P.n_chunks);
  const int hq = params->hq, hkv = params->hkv, d = params->d;
  if (hq <= 0 || hkv <= 0 || hq % hkv) return fail(TREE_ERR_UNSUPPORTED, "tree_attn_fwd: hq %d, hkv %d", hq, hkv);
  if (d != 64 && d != 128) return fail(TREE_ERR_UNSUPPORTED, "tree_attn_fwd: head dim %d not in {64, 128}", d);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(plan_dev))
    return fail(TREE_ERR_UNSUPPORTED, "tree_attn_fwd: tensors must be 16-byte aligned");
  if (params->work && (reinterpret_cast<uintptr_t>(params->work) & 7))
    return fail(TREE_ERR_UNSUPPORTED, "tree_attn_fwd: work counter must be 8-byte aligned");
  const float scale = params->scale > 0.f ? params->scale : 1.f / std::sqrt((float)d);
  const int32_t *img = reinterpret_cast<const int32_t *>(plan_dev);
  const cudaStream_t s = as_stream(stream);
  const bool pair = (hq / hkv) % 2 == 0;
  if (P.pack_heads > 1 && hq / hkv != P.pack_heads)
    return fail(TREE_ERR_UNSUPPORTED, "tree_attn_fwd: the plan packs %d q heads per kv head, the launch has %d / %d",
                P.pack_heads, hq, hkv);
  if (d == 64)
    return pair ? launch_tc<64, 2>(P, img, chunk, q, k, v, o, lse, hq, hkv, scale, params->work, params->self_test, status, s)
                : launch_tc<64, 1>(P, img, chunk, q, k, v, o, lse, hq, hkv, scale, params->work, params->self_test, status, s);
  return pair ? launch_tc<128, 2>(P, img, chunk, q, k, v, o, lse, hq, hkv, scale, params->work, params->self_test, status, s)
              : launch_tc<128, 1>(P, img, chunk, q, k, v, o, lse, hq, hkv, scale, params->work, params->self_test, status, s);
}

// ---------------------------------------------------------------------------
// tree_attn_fwd_noalloc: the same attention for callers that cannot allocate
// device memory themselves.  The persistent CTAs' work counter (two int32 per
// chunk) then lives in this file's own device array instead of in caller
// memory.  The array holds kNoAllocChunks counter pairs and stays resident on
// every device that loads the library until the process exits.

namespace tree {
namespace {

constexpr int kNoAllocChunks = 256;
static __device__ __align__(256) int32_t g_noalloc_work[2 * kNoAllocChunks];

constexpr int kMaxDevices = 64;
struct NoAllocSlot {
  unsigned long long ctx_id;  // context the address belongs to (0: none yet)
  int32_t *ptr;
};
NoAllocSlot g_noalloc_slot[kMaxDevices] = {};
std::mutex g_noalloc_mutex;

// Unique id of the calling thread's current CUDA context, 0 if there is none
// (ids are never reused within a process, unlike context handles).
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the array in the current context.  Looked up on the
// first call on a device and again whenever the device's context has changed
// since (after cudaDeviceReset, say, the old address belongs to a context
// that no longer exists).
int noalloc_counters(int32_t **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_attn_fwd_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(TREE_ERR_UNSUPPORTED, "tree_attn_fwd_noalloc: device %d beyond %d", dev, kMaxDevices);
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoAllocSlot &slot = g_noalloc_slot[dev];
  if (ctx == 0 || slot.ctx_id != ctx || !slot.ptr) {
    int32_t *ptr = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void **>(&ptr), g_noalloc_work);
    if (e != cudaSuccess || !ptr)
      return fail(TREE_ERR_CUDA, "tree_attn_fwd_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    slot.ptr = ptr;
    slot.ctx_id = current_context_id();  // the lookup has made the device's context current
  }
  *out = slot.ptr;
  return TREE_OK;
}

}  // namespace
}  // namespace tree

extern "C" TREE_API int tree_attn_fwd_noalloc(const tree_plan_t *plan, const void *plan_dev, int32_t chunk,
                                              const void *q, const void *k, const void *v, void *o, float *lse,
                                              const tree_attn_params_t *params, int32_t *status,
                                              tree_stream_t stream) {
  using namespace tree;
  if (!plan || !params) return fail(TREE_ERR_INVALID_ARG, "tree_attn_fwd_noalloc: NULL argument");
  if (params->work)
    return fail(TREE_ERR_INVALID_ARG, "tree_attn_fwd_noalloc: params->work must be NULL (the counters are built in)");
  if (plan->p.n_chunks > kNoAllocChunks)
    return fail(TREE_ERR_UNSUPPORTED, "tree_attn_fwd_noalloc: plan has %d chunks; the built-in counters cover %d",
                plan->p.n_chunks, kNoAllocChunks);
  if (chunk < 0 || chunk >= plan->p.n_chunks)
    return fail(TREE_ERR_INVALID_ARG, "tree_attn_fwd_noalloc: chunk %d out of range [0, %d)", chunk, plan->p.n_chunks);
  int32_t *counters = nullptr;
  int rc = noalloc_counters(&counters);
  if (rc != TREE_OK) return rc;
  int32_t *work = counters + 2 * chunk;
  // start from zero whatever an earlier call left behind
  const cudaError_t e = cudaMemsetAsync(work, 0, 2 * sizeof(int32_t), as_stream(stream));
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_attn_fwd_noalloc: %s", cudaGetErrorString(e));
  tree_attn_params_t p = *params;
  p.work = work;
  return tree_attn_fwd(plan, plan_dev, chunk, q, k, v, o, lse, &p, status, stream);
}
