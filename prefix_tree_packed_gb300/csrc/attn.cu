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
//       it.  These warps raise their register budget to 208 (setmaxnreg).
//   producer warp: TMA loads of the Q tiles and of K, V (plus the 128 subtree
//       ends of the key tile) into a ring of shared-memory stages.
//   MMA warp: one thread issues tcgen05.mma: S_h = Q_h K^T (A, B in shared
//       memory, 128 x 128 x d) and O_h += P_h V (A = P_h in tensor memory,
//       B = V in shared memory, 128 x d x 128), each followed by a commit to an
//       mbarrier.  The producer/MMA warpgroup lowers its budget to 88 registers.
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

#include <cmath>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm103.cuh"

namespace tree {
namespace {

using namespace sm103;

constexpr int BN = 128;                    // keys per tile (queries per tile: 128, one per TMEM lane)
constexpr uint32_t BOX_BYTES = 128 * 128;  // one 128-row x 64-column f16 box (128-byte rows)
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 500000000ull;

struct AttnArgs {
  const int32_t *send;
  const QTile *qtiles;
  const int32_t *ent;
  const int32_t *order;
  __half *o;
  float *lse;
  int32_t *status;
  int32_t t0, q0, n_tot, hq, hkv, ratio;
  float scale_log2;
};

template <int D, int NH>
struct Cfg {
  static constexpr int CB = D / 64;               // 64-column boxes per row of a tile
  static constexpr int STAGES = D == 64 ? 3 : 2;  // K/V ring depth
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + NH * CB * BOX_BYTES;
  static constexpr uint32_t V_OFF = K_OFF + STAGES * CB * BOX_BYTES;
  static constexpr uint32_t SEND_OFF = V_OFF + STAGES * CB * BOX_BYTES;
  static constexpr uint32_t SMEM = SEND_OFF + STAGES * 512 + 1024;  // + alignment slack
  static constexpr int WARPS = 4 * NH + 4;        // softmax warpgroups + producer/MMA warpgroup
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int PROD_WARP = 4 * NH;
  static constexpr int MMA_WARP = 4 * NH + 1;
  static constexpr bool PSEP = D == 64;           // P in its own columns
  static constexpr uint32_t P_COL = 128 * NH;     // P_h at P_COL + 64h (PSEP only)
  static constexpr uint32_t O_COL = PSEP ? 128 * NH + 64 * NH : 128 * NH;
  static constexpr uint32_t TMEM_USED = O_COL + D * NH;
  static constexpr uint32_t TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
  // 12 warps launch at 168 registers (3 per SM sub-partition of 16384); setmaxnreg moves them
  static constexpr int SOFTMAX_REGS = 208;       // 2 x 208 + 88 = 504 <= 512 per sub-partition
  static constexpr int SERVICE_REGS = 88;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[3], v_full[3], kv_empty[3];
  uint64_t s_full[2], s_free[2], p_full[2], o_done[2];
  uint32_t tmem;
  int32_t abort;
};

// Wait for the phase with the given parity; false (and the CTA's abort flag
// set) if it has not completed within limit_ns, or, with honor_abort, as soon
// as another thread of the CTA has given up.
TREE_DEV bool wait_bar(uint32_t bar, uint32_t parity, volatile int32_t *abort, int32_t *status,
                       bool honor_abort = true, uint64_t limit_ns = kWaitNs) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
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

// Warp-uniform form for the softmax warps, whose next steps are warp-collective.
TREE_DEV bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int32_t *abort, int32_t *status) {
  const bool ok = wait_bar(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok);
}

template <int D, int NH>
__global__ void __launch_bounds__(Cfg<D, NH>::THREADS, 1)
    tree_attn_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, const AttnArgs a) {
  using C = Cfg<D, NH>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(sm);
  const int32_t *sSend = reinterpret_cast<const int32_t *>(sm + C::SEND_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pairs = a.ratio / NH;
  const int per_tile = a.hkv * pairs;
  const int rank = blockIdx.x / per_tile;
  const int rem = blockIdx.x - rank * per_tile;
  const int g = rem / pairs;
  const int h0 = g * a.ratio + (rem - g * pairs) * NH;
  const QTile qt = a.qtiles[__ldg(a.order + a.t0 + rank)];
  const int n = qt.ent1 - qt.ent0;
  volatile int32_t *abort = &bars.abort;

  const uint32_t b_q = smem_u32(&bars.q_full);
  auto b_k = [&](int s) { return smem_u32(&bars.k_full[s]); };
  auto b_v = [&](int s) { return smem_u32(&bars.v_full[s]); };
  auto b_e = [&](int s) { return smem_u32(&bars.kv_empty[s]); };
  auto b_s = [&](int h) { return smem_u32(&bars.s_full[h]); };
  auto b_f = [&](int h) { return smem_u32(&bars.s_free[h]); };
  auto b_p = [&](int h) { return smem_u32(&bars.p_full[h]); };
  auto b_o = [&](int h) { return smem_u32(&bars.o_done[h]); };

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(b_k(s), 1);
      mbar_init(b_v(s), 1);
      mbar_init(b_e(s), 1);
    }
    for (int h = 0; h < NH; ++h) {
      mbar_init(b_s(h), 1);
      mbar_init(b_f(h), 128);
      mbar_init(b_p(h), 128);
      mbar_init(b_o(h), 1);
    }
    bars.abort = 0;
    mbar_fence_init();
  }
  if (warp == C::MMA_WARP) tmem_alloc(smem_u32(&bars.tmem), C::TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = bars.tmem;

  if (warp >= 4 * NH) {
    if (NH == 2) regs_dec<C::SERVICE_REGS>();
    if (warp == C::PROD_WARP && n > 0) {
      // ---------------------------------------------------------- producer (whole warp, one lane issues)
      if (elect_one()) {
        prefetch_map(&mq);
        prefetch_map(&mk);
        prefetch_map(&mv);
        mbar_expect_tx(b_q, NH * C::CB * BOX_BYTES);
#pragma unroll
        for (int h = 0; h < NH; ++h)
#pragma unroll
          for (int c = 0; c < C::CB; ++c)
            tma_load_2d(s_base + C::Q_OFF + (h * C::CB + c) * BOX_BYTES, &mq, (h0 + h) * D + 64 * c, qt.row0 - a.q0,
                        b_q);
      }
      __syncwarp();
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int st = i % C::STAGES;
        if (i >= C::STAGES && !wait_bar_warp(b_e(st), ((i / C::STAGES) - 1) & 1, abort, a.status)) break;
        const int j0 = (__ldg(a.ent + qt.ent0 + i) >> 1) * BN;
        if (elect_one()) {
          mbar_expect_tx(b_k(st), C::CB * BOX_BYTES + 512);
#pragma unroll
          for (int c = 0; c < C::CB; ++c)
            tma_load_2d(s_base + C::K_OFF + (st * C::CB + c) * BOX_BYTES, &mk, g * D + 64 * c, j0, b_k(st));
          bulk_load(s_base + C::SEND_OFF + st * 512, a.send + j0, 512, b_k(st));
          mbar_expect_tx(b_v(st), C::CB * BOX_BYTES);
#pragma unroll
          for (int c = 0; c < C::CB; ++c)
            tma_load_2d(s_base + C::V_OFF + (st * C::CB + c) * BOX_BYTES, &mv, g * D + 64 * c, j0, b_v(st));
        }
        __syncwarp();
        issued = i + 1;
      }
      // wind down: every copy issued must have landed before the CTA exits
      wait_bar(b_q, 0, abort, nullptr, false, kDrainNs);
      for (int i = (issued > C::STAGES ? issued - C::STAGES : 0); i < issued; ++i) {
        wait_bar(b_k(i % C::STAGES), (i / C::STAGES) & 1, abort, nullptr, false, kDrainNs);
        wait_bar(b_v(i % C::STAGES), (i / C::STAGES) & 1, abort, nullptr, false, kDrainNs);
      }
    } else if (warp == C::MMA_WARP && n > 0) {
      // ---------------------------------------------------------- MMA issuer (whole warp, one lane issues)
      constexpr uint32_t idesc_qk = idesc_f16(128, 128, false);
      constexpr uint32_t idesc_pv = idesc_f16(128, D, true);
      auto issue_qk = [&](int h, int st) {
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
            const uint64_t da = sdesc_sw128(s_base + C::Q_OFF + h * C::CB * BOX_BYTES + off, 16, 1024);
            const uint64_t db = sdesc_sw128(s_base + C::K_OFF + st * C::CB * BOX_BYTES + off, 16, 1024);
            mma_ss(tmem + 128 * h, da, db, idesc_qk, kk > 0);
          }
          mma_commit(b_s(h));
        }
        __syncwarp();
      };
      auto issue_pv = [&](int h, int st, int i) {
        const uint32_t p_col = C::PSEP ? C::P_COL + 64 * h : 128 * h;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t db =
                sdesc_sw128(s_base + C::V_OFF + st * C::CB * BOX_BYTES + kk * 2048, BOX_BYTES, 1024);
            mma_ts(tmem + C::O_COL + D * h, tmem + p_col + 8 * kk, db, idesc_pv, (i > 0 || kk > 0));
          }
          mma_commit(b_o(h));
        }
        __syncwarp();
      };
      bool ok = wait_bar_warp(b_q, 0, abort, a.status) && wait_bar_warp(b_k(0), 0, abort, a.status);
      int last_o = -1, last_h = 0;  // iteration and head of the last PV commit issued
      if (ok) {
        fence_after();
        for (int h = 0; h < NH; ++h) issue_qk(h, 0);
        for (int i = 0; i < n && ok; ++i) {
          const int st = i % C::STAGES;
          const int st2 = (i + 1) % C::STAGES;
          if (C::PSEP) {
            // next S first: S_h is free once the softmax has read it into registers
            if (i + 1 < n) {
              if (!(ok = wait_bar_warp(b_k(st2), ((i + 1) / C::STAGES) & 1, abort, a.status))) break;
              for (int h = 0; h < NH && ok; ++h) {
                if (!(ok = wait_bar_warp(b_f(h), i & 1, abort, a.status))) break;
                fence_after();
                issue_qk(h, st2);
              }
              if (!ok) break;
            }
            if (!(ok = wait_bar_warp(b_v(st), (i / C::STAGES) & 1, abort, a.status))) break;
            for (int h = 0; h < NH && ok; ++h) {
              if (!(ok = wait_bar_warp(b_p(h), i & 1, abort, a.status))) break;
              fence_after();
              issue_pv(h, st, i);
              last_o = i;
              last_h = h;
            }
            if (ok && i + C::STAGES < n) {
              if (elect_one()) mma_commit(b_e(st));
              __syncwarp();
            }
          } else {
            // P_h shares S_h's columns: per head, PV(i) then (once it is done) S(i+1)
            if (!(ok = wait_bar_warp(b_v(st), (i / C::STAGES) & 1, abort, a.status))) break;
            for (int h = 0; h < NH && ok; ++h) {
              if (!(ok = wait_bar_warp(b_p(h), i & 1, abort, a.status))) break;
              fence_after();
              issue_pv(h, st, i);
              last_o = i;
              last_h = h;
              if (h == NH - 1 && i + C::STAGES < n) {
                if (elect_one()) mma_commit(b_e(st));
                __syncwarp();
              }
              if (i + 1 < n) {
                if (h == 0 && !(ok = wait_bar_warp(b_k(st2), ((i + 1) / C::STAGES) & 1, abort, a.status))) break;
                if (!(ok = wait_bar_warp(b_o(h), i & 1, abort, a.status))) break;
                fence_after();
                issue_qk(h, st2);
              }
            }
          }
        }
      }
      // wind down: all issued MMAs complete before tensor memory is freed
      if (last_o >= 0) wait_bar(b_o(last_h), last_o & 1, abort, nullptr, false, kDrainNs);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    if (NH == 2) regs_inc<C::SOFTMAX_REGS>();
    const int h = warp >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int iq = qt.row0 + r;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t tS = t_lane + 128 * h;
    const uint32_t tP = C::PSEP ? t_lane + C::P_COL + 64 * h : tS;
    const uint32_t tO = t_lane + C::O_COL + D * h;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    int done = 0;
    for (int i = 0; i < n; ++i) {
      const int st = i % C::STAGES;
      const int e = __ldg(a.ent + qt.ent0 + i);
      if (!(ok = wait_bar_warp(b_s(h), i & 1, abort, a.status))) break;
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
      if (e & 1) {
        // partial tile: key j = j0 + c is visible iff j <= iq < send[j]
        if (!(ok = wait_bar_warp(b_k(st), (i / C::STAGES) & 1, abort, a.status))) break;
        const int cmax = iq - (e >> 1) * BN;  // keys c <= cmax are not after the query
        const int4 *sd = reinterpret_cast<const int4 *>(sSend + st * 128);
#pragma unroll
        for (int c4 = 0; c4 < 32; ++c4) {
          const int4 se = sd[c4];
          const int sv[4] = {se.x, se.y, se.z, se.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = 4 * c4 + u;
            if (!((c <= cmax) && (iq < sv[u]))) s[c] = __float_as_uint(-INFINITY);
          }
        }
      }
      float mx8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx8[u] = __uint_as_float(s[u]);
#pragma unroll
      for (int c = 8; c < 128; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], __uint_as_float(s[c]));
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float mt = mx * a.scale_log2;  // -inf stays -inf (scale > 0)
      const bool grow = mt > m + 8.f;      // also true for the first finite maximum
      float alpha = 1.f;
      if (grow) {
        alpha = ex2(m - mt);  // 0 when m is -inf
        m = mt;
      }
      const float mu = (m == -INFINITY) ? 0.f : m;
      float sum8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) sum8[u] = 0.f;
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        const float p0 = ex2(fmaf(__uint_as_float(s[c]), a.scale_log2, -mu));
        const float p1 = ex2(fmaf(__uint_as_float(s[c + 1]), a.scale_log2, -mu));
        sum8[(c >> 1) & 7] += p0 + p1;
        s[c >> 1] = pack_f16x2(p0, p1);
      }
      l = l * alpha + (((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7])));
      // PV_h(i-1) must be done before P_h is rewritten (separate P) or O_h is rescaled
      const bool need_o = i > 0 && __any_sync(0xffffffffu, grow);
      if (i > 0 && (C::PSEP || need_o)) {
        if (!(ok = wait_bar_warp(b_o(h), (i - 1) & 1, abort, a.status))) break;
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
      done = i + 1;
    }
    // ---- epilogue: O / l -> f16 rows of the chunk's output
    if (ok && done == n && n > 0 && wait_bar_warp(b_o(h), (n - 1) & 1, abort, a.status)) {
      fence_after();
      const bool valid = iq < qt.row1;
      const float inv = 1.f / l;
      __half *dst = a.o + ((size_t)(iq - a.q0) * a.hq + (h0 + h)) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = pack_f16x2(__uint_as_float(o[2 * u]) * inv, __uint_as_float(o[2 * u + 1]) * inv);
        if (valid) {
          uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
          for (int u = 0; u < 4; ++u) d4[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      if (valid && a.lse) {
        const float mu = (m == -INFINITY) ? 0.f : m;
        a.lse[(size_t)(iq - a.q0) * a.hq + h0 + h] = (mu + __log2f(l)) * 0.69314718055994531f;
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D map over a [rows, cols] f16 matrix with 128-row x 64-column boxes, 128-byte swizzle.
int make_map(CUtensorMap *map, const void *base, int64_t cols, int64_t rows) {
  auto enc = encode_fn();
  if (!enc) return fail(TREE_ERR_CUDA, "tree_attn_fwd: cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TREE_ERR_CUDA, "tree_attn_fwd: tensor map encode failed (%d)", (int)r);
  return TREE_OK;
}

template <int D, int NH>
int launch_tc(const Plan &P, const int32_t *img, int chunk, const void *q, const void *k, const void *v, void *o,
              float *lse, int hq, int hkv, float scale, int32_t *status, cudaStream_t s) {
  using C = Cfg<D, NH>;
  static bool attr_set = false;
  auto kern = tree_attn_tc<D, NH>;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_attn_fwd: %s", cudaGetErrorString(e));
    attr_set = true;
  }
  const int32_t q0 = P.chunk_q0[chunk], nq = P.chunk_q1[chunk] - q0;
  CUtensorMap mq, mk, mv;
  int rc;
  if ((rc = make_map(&mq, q, (int64_t)hq * D, nq)) || (rc = make_map(&mk, k, (int64_t)hkv * D, P.n_tot)) ||
      (rc = make_map(&mv, v, (int64_t)hkv * D, P.n_tot)))
    return rc;
  AttnArgs a;
  a.send = img + P.off_send;
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
  const int tiles = P.chunk_t1[chunk] - P.chunk_t0[chunk];
  const dim3 grid((unsigned)(tiles * hkv * (a.ratio / NH)));
  kern<<<grid, C::THREADS, C::SMEM, s>>>(mq, mk, mv, a);
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
  const float scale = params->scale > 0.f ? params->scale : 1.f / std::sqrt((float)d);
  const int32_t *img = reinterpret_cast<const int32_t *>(plan_dev);
  const cudaStream_t s = as_stream(stream);
  const bool pair = (hq / hkv) % 2 == 0;
  if (d == 64)
    return pair ? launch_tc<64, 2>(P, img, chunk, q, k, v, o, lse, hq, hkv, scale, status, s)
                : launch_tc<64, 1>(P, img, chunk, q, k, v, o, lse, hq, hkv, scale, status, s);
  return pair ? launch_tc<128, 2>(P, img, chunk, q, k, v, o, lse, hq, hkv, scale, status, s)
              : launch_tc<128, 1>(P, img, chunk, q, k, v, o, lse, hq, hkv, scale, status, s);
}
