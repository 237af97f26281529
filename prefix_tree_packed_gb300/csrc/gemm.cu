// tree_gemm: the projections of a Llama layer around the tree attention,
// C = epilogue(A B^T) with A an activation [M, K] and B a Linear weight
// [N, K] (both f16, K contiguous), f32 accumulation in tensor memory, C f16.
// The basal-rs Architecture page ("01 / Request path: GPU forward pass") runs
// the Llama model in f16 over the batch as one compact token list; its GEMMs
// have no split over K here, so every output is one f32 sum in a fixed order.
//
// Epilogues (fused, per output element):
//   STORE     C = A B^T
//   RESIDUAL  C = A B^T + R            (R f16 [M, N], may be C itself)
//   SWIGLU    C = silu(A G^T) * (A U^T), B = [G; U] with 2N rows,
//             silu(g) = g / (1 + e^-g)  (the Llama MLP gate)
//   STORE_F32 C = A B^T kept in f32 (the letter logits of the final layer)
//
// Work decomposition: persistent CTAs (one per SM) walk 128 x 256 output
// tiles (SWIGLU: 128 x 128 outputs from 128 gate + 128 up columns) in an
// M-grouped order.  Roles: a producer warp (TMA loads of 64-wide K slices of
// A and B into a 4-stage shared-memory ring), an MMA warp (one elected lane
// issues tcgen05.mma M=128 N=256 K=16, the accumulator double-buffered in
// tensor memory, 2 x 256 columns) and four epilogue warps (tcgen05.ld of their
// 32 rows, epilogue in f32, f16 stores) that drain tile t while the MMAs of
// tile t + 1 run.  Every mbarrier wait is bounded: after ~2 s it sets
// TREE_ERR_TIMEOUT in the status word and the CTA winds down.

#include <cmath>

#include "common.cuh"
#include "sm103.cuh"
#include "tree_layer.h"

namespace tree {
namespace {

using namespace sm103;

constexpr int GBM = 128, GBK = 64;
constexpr uint32_t G_A_BYTES = GBM * GBK * 2;  // 16 KB
constexpr int G_THREADS = 192;                  // producer, MMA, 4 epilogue warps
constexpr int G_MAX_STAGES = 8;

// Tile width BN = the MMA's N: 256 (large m: few, long tiles) or 64 (small m:
// enough tiles to spread the weight reads over the SMs).  Either way every
// output is the same f32 sum over K in the same order.
template <int BN>
struct GCfg {
  static constexpr uint32_t B_BYTES = BN * GBK * 2;
  static constexpr uint32_t STAGE = G_A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 4 : 8;
  static constexpr uint32_t SMEM = STAGES * STAGE + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 2 * BN;             // two accumulators
};
constexpr int G_GROUP_M = 16;                           // M tiles per raster group
constexpr uint64_t kGemmWaitNs = 2000000000ull;
constexpr uint64_t kGemmDrainNs = 500000000ull;

constexpr int kEpiQKV = 16;  // internal: STORE with the columns split over three outputs (tree_gemm_qkv)

struct GemmArgs {
  int m, n, k;         // C is m x n; B has n rows (2n for SWIGLU)
  int n1, n2;          // kEpiQKV: columns [0, n1) -> c, [n1, n1 + n2) -> c2, [n1 + n2, n) -> c3
  __half *c2, *c3;
  int tiles_m, tiles_n, n_tiles, nk;
  int bn;              // output columns per tile (256, SWIGLU 128)
  int epi;
  __half *c;
  const __half *r;
  int32_t *status;
};

struct GBars {
  uint64_t full[G_MAX_STAGES], empty[G_MAX_STAGES], acc_full[2], acc_empty[2];
  uint32_t tmem;
  int32_t abort;
};

__device__ bool gwait(uint32_t bar, uint32_t parity, volatile int32_t *abort, int32_t *status,
                      uint64_t limit_ns = kGemmWaitNs, bool honor_abort = true) {
  if (mbar_test(bar, parity)) return true;
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

__device__ __forceinline__ bool gwait_warp(uint32_t bar, uint32_t parity, volatile int32_t *abort, int32_t *status) {
  return __all_sync(0xffffffffu, gwait(bar, parity, abort, status));
}

// Tile t -> (tile_m, tile_n): groups of G_GROUP_M row tiles, columns outer
// within a group, so that concurrently running CTAs share A rows and B columns in L2.
__device__ __forceinline__ void tile_of(const GemmArgs &a, int t, int &tm, int &tn) {
  const int per_group = G_GROUP_M * a.tiles_n;
  const int g = t / per_group;
  const int first = g * G_GROUP_M;
  const int rows = min(a.tiles_m - first, G_GROUP_M);
  const int in = t - g * per_group;
  tm = first + in % rows;
  tn = in / rows;
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + __expf(-g)); }

template <int BN>
__global__ void __launch_bounds__(G_THREADS, 1)
    gemm_tc(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb, const GemmArgs a) {
  using Cf = GCfg<BN>;
  constexpr int GSTAGES = Cf::STAGES;
  constexpr uint32_t G_STAGE = Cf::STAGE;
  constexpr uint32_t G_B_BYTES = Cf::B_BYTES;
  extern __shared__ uint8_t g_smem_raw[];
  __shared__ GBars bars;
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(g_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int32_t *abort = &bars.abort;
  auto b_full = [&](int s) { return smem_u32(&bars.full[s]); };
  auto b_empty = [&](int s) { return smem_u32(&bars.empty[s]); };
  auto b_af = [&](int b) { return smem_u32(&bars.acc_full[b]); };
  auto b_ae = [&](int b) { return smem_u32(&bars.acc_empty[b]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < GSTAGES; ++s) {
      mbar_init(b_full(s), 1);
      mbar_init(b_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(b_af(b), 1);
      mbar_init(b_ae(b), 128);
    }
    bars.abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&bars.tmem), Cf::TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = bars.tmem;
  griddep_wait();  // A (and R) may come from the kernel before this one in the stream

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      prefetch_map(&ma);
      prefetch_map(&mb);
    }
    __syncwarp();
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < a.n_tiles && ok; t += gridDim.x) {
      int tm, tn;
      tile_of(a, t, tm, tn);
      const int m0 = tm * GBM, n0 = tn * a.bn;
      const int nb2 = a.epi == TREE_GEMM_SWIGLU ? a.n + n0 : n0 + BN / 2;  // rows of the second B box
      for (int kb = 0; kb < a.nk; ++kb, ++it) {
        const int s = it % GSTAGES;
        if (it >= GSTAGES && !(ok = gwait_warp(b_empty(s), ((it / GSTAGES) - 1) & 1, abort, a.status))) break;
        if (elect_one()) {
          const uint32_t st = s_base + s * G_STAGE;
          mbar_expect_tx(b_full(s), G_STAGE);
          tma_load_2d(st, &ma, kb * GBK, m0, b_full(s));
          tma_load_2d(st + G_A_BYTES, &mb, kb * GBK, n0, b_full(s));
          tma_load_2d(st + G_A_BYTES + G_B_BYTES / 2, &mb, kb * GBK, nb2, b_full(s));
        }
        __syncwarp();
      }
    }
    griddep_launch();
    // wind down: every load issued has landed
    for (int u = (it > GSTAGES ? it - GSTAGES : 0); u < it; ++u)
      gwait(b_full(u % GSTAGES), (u / GSTAGES) & 1, abort, nullptr, kGemmDrainNs, false);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_f16(GBM, BN, false);
    int it = 0, tc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < a.n_tiles && ok; t += gridDim.x, ++tc) {
      const int b = tc & 1;
      if (tc >= 2 && !(ok = gwait_warp(b_ae(b), ((tc / 2) - 1) & 1, abort, a.status))) break;
      fence_after();
      const uint32_t d = tmem + (uint32_t)(b * BN);
      for (int kb = 0; kb < a.nk; ++kb, ++it) {
        const int s = it % GSTAGES;
        if (!(ok = gwait_warp(b_full(s), (it / GSTAGES) & 1, abort, a.status))) break;
        fence_after();
        const uint32_t st = s_base + s * G_STAGE;
        const uint64_t da = sdesc_sw128(st, 16, 1024), db = sdesc_sw128(st + G_A_BYTES, 16, 1024);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < GBK / 16; ++kk) mma_ss(d, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) != 0);
          mma_commit(b_empty(s));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) mma_commit(b_af(b));
      __syncwarp();
    }
    // wind down: every MMA issued has completed
    if (it > 0) {
      const int u = it - 1;
      gwait(b_empty(u % GSTAGES), (u / GSTAGES) & 1, abort, nullptr, kGemmDrainNs, false);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int qd = warp & 3;  // tensor-memory lane quarter of this warp
    const uint32_t t_lane = tmem + ((uint32_t)(32 * qd) << 16);
    int tc = 0;
    for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x, ++tc) {
      const int b = tc & 1;
      int tm, tn;
      tile_of(a, t, tm, tn);
      const int row = tm * GBM + 32 * qd + lane, n0 = tn * a.bn;
      const bool row_ok = row < a.m;
      // the residual row is read before the accumulator is ready: its loads are all
      // in flight while the tile's last MMAs run
      uint4 res[BN / 8];
      if (a.epi == TREE_GEMM_RESIDUAL) {
        const __half *rrow = a.r + (size_t)row * a.n;
#pragma unroll
        for (int u = 0; u < BN / 8; ++u) {
          const int c = n0 + 8 * u;
          res[u] = (row_ok && c < a.n) ? *reinterpret_cast<const uint4 *>(rrow + c) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (!gwait_warp(b_af(b), (tc / 2) & 1, abort, a.status)) break;
      fence_after();
      __half *crow = a.c + (size_t)row * a.n;
      const uint32_t acc = t_lane + (uint32_t)(b * BN);
      if (a.epi == TREE_GEMM_SWIGLU) {
        for (int ch = 0; ch < BN / 64; ++ch) {
          uint32_t g[32], u[32];
          tmem_ld32(acc + 32 * ch, g);
          tmem_ld32(acc + BN / 2 + 32 * ch, u);
          tmem_wait_ld();
          const int c0 = n0 + 32 * ch;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            uint32_t *wp = &w.x;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = 8 * v + 2 * e;
              wp[e] = pack_f16x2(silu(__uint_as_float(g[j])) * __uint_as_float(u[j]),
                                 silu(__uint_as_float(g[j + 1])) * __uint_as_float(u[j + 1]));
            }
            if (row_ok && c0 + 8 * v < a.n) *reinterpret_cast<uint4 *>(crow + c0 + 8 * v) = w;
          }
        }
      } else {
#pragma unroll
        for (int ch = 0; ch < BN / 32; ++ch) {
          uint32_t x[32];
          tmem_ld32(acc + 32 * ch, x);
          tmem_wait_ld();
          const int c0 = n0 + 32 * ch;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int c = c0 + 8 * v;
            if (!row_ok || c >= a.n) continue;
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(x[8 * v + e]);
            if (a.epi == TREE_GEMM_RESIDUAL) {
              const __half2 *rh = reinterpret_cast<const __half2 *>(&res[4 * ch + v]);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 r2 = __half22float2(rh[e]);
                f[2 * e] += r2.x;
                f[2 * e + 1] += r2.y;
              }
            }
            if (a.epi == TREE_GEMM_STORE_F32) {
              float *frow = reinterpret_cast<float *>(a.c) + (size_t)row * a.n + c;
              reinterpret_cast<float4 *>(frow)[0] = make_float4(f[0], f[1], f[2], f[3]);
              reinterpret_cast<float4 *>(frow)[1] = make_float4(f[4], f[5], f[6], f[7]);
              continue;
            }
            uint4 w;
            w.x = pack_f16x2(f[0], f[1]);
            w.y = pack_f16x2(f[2], f[3]);
            w.z = pack_f16x2(f[4], f[5]);
            w.w = pack_f16x2(f[6], f[7]);
            __half *dst = crow + c;
            if (a.epi == kEpiQKV)
              dst = c < a.n1 ? a.c + (size_t)row * a.n1 + c
                             : (c < a.n1 + a.n2 ? a.c2 + (size_t)row * a.n2 + (c - a.n1)
                                                : a.c3 + (size_t)row * a.n2 + (c - a.n1 - a.n2));
            *reinterpret_cast<uint4 *>(dst) = w;
          }
        }
      }
      fence_before();
      mbar_arrive(b_ae(b));
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, Cf::TMEM_COLS);
  }
}

}  // namespace
}  // namespace tree

namespace tree {
namespace {

template <int BN>
int launch_gemm(const void *a, const void *b, void *c, const void *r, int32_t m, int32_t n, int32_t k, int32_t epi,
                int32_t *status, cudaStream_t s, int32_t n1 = 0, int32_t n2 = 0, void *c2 = nullptr,
                void *c3 = nullptr) {
  using Cf = GCfg<BN>;
  int rc = set_max_dynamic_smem(reinterpret_cast<const void *>(gemm_tc<BN>), (int)Cf::SMEM, "tree_gemm");
  if (rc) return rc;
  const int nb_rows = epi == TREE_GEMM_SWIGLU ? 2 * n : n;
  CUtensorMap ma, mb;
  if ((rc = make_map(&ma, a, k, m, "tree_gemm")) || (rc = make_map(&mb, b, k, nb_rows, "tree_gemm", BN / 2))) return rc;
  GemmArgs g;
  g.m = m;
  g.n = n;
  g.k = k;
  g.bn = epi == TREE_GEMM_SWIGLU ? BN / 2 : BN;
  g.tiles_m = (m + GBM - 1) / GBM;
  g.tiles_n = (n + g.bn - 1) / g.bn;
  g.n_tiles = g.tiles_m * g.tiles_n;
  g.nk = (k + GBK - 1) / GBK;
  g.epi = epi;
  g.c = reinterpret_cast<__half *>(c);
  g.r = reinterpret_cast<const __half *>(r);
  g.status = status;
  g.n1 = n1;
  g.n2 = n2;
  g.c2 = reinterpret_cast<__half *>(c2);
  g.c3 = reinterpret_cast<__half *>(c3);
  const dim3 grid((unsigned)std::min(g.n_tiles, sm_count()));
  const cudaError_t e = launch_dependent(gemm_tc<BN>, grid, dim3(G_THREADS), Cf::SMEM, s, ma, mb, g);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_gemm: launch failed: %s", cudaGetErrorString(e));
  return launch_status("tree_gemm");
}

// Narrow tiles for at most three row tiles (a single request, the readout rows):
// there the weights' reads dominate and 64-column tiles spread them over more
// SMs.  From four row tiles on, and for the SwiGLU projection at any m, wide
// tiles measured faster (Llama-1B shapes: down at m = 300 32 vs 39 us narrow
// first, at m = 600 60 vs 40 us wide first).
bool narrow_tiles(int32_t m, int32_t epi) { return (m + GBM - 1) / GBM <= 3 && epi != TREE_GEMM_SWIGLU; }

}  // namespace
}  // namespace tree

extern "C" TREE_API int tree_gemm_ex(const void *a, const void *b, void *c, const void *r, int32_t m, int32_t n,
                                     int32_t k, int32_t epi, int32_t tile_n, int32_t *status, tree_stream_t stream) {
  using namespace tree;
  if (!a || !b || !c) return fail(TREE_ERR_INVALID_ARG, "tree_gemm: NULL argument");
  if (m < 0 || n <= 0 || k <= 0) return fail(TREE_ERR_INVALID_ARG, "tree_gemm: m %d, n %d, k %d", m, n, k);
  if (epi != TREE_GEMM_STORE && epi != TREE_GEMM_RESIDUAL && epi != TREE_GEMM_SWIGLU && epi != TREE_GEMM_STORE_F32)
    return fail(TREE_ERR_INVALID_ARG, "tree_gemm: unknown epilogue %d", epi);
  if (epi == TREE_GEMM_RESIDUAL && !r) return fail(TREE_ERR_INVALID_ARG, "tree_gemm: RESIDUAL needs r");
  if (tile_n != 0 && tile_n != 64 && tile_n != 256)
    return fail(TREE_ERR_INVALID_ARG, "tree_gemm: tile_n %d not in {0, 64, 256}", tile_n);
  if (n % 8 || k % 8) return fail(TREE_ERR_UNSUPPORTED, "tree_gemm: n %d and k %d must be multiples of 8", n, k);
  if (!aligned16(a) || !aligned16(b) || !aligned16(c) || (r && !aligned16(r)))
    return fail(TREE_ERR_UNSUPPORTED, "tree_gemm: tensors must be 16-byte aligned");
  if (m == 0) return TREE_OK;
  if (tile_n == 0) tile_n = narrow_tiles(m, epi) ? 64 : 256;
  const cudaStream_t s = as_stream(stream);
  return tile_n == 256 ? launch_gemm<256>(a, b, c, r, m, n, k, epi, status, s)
                       : launch_gemm<64>(a, b, c, r, m, n, k, epi, status, s);
}

extern "C" TREE_API int tree_gemm(const void *a, const void *b, void *c, const void *r, int32_t m, int32_t n,
                                  int32_t k, int32_t epi, int32_t *status, tree_stream_t stream) {
  return tree_gemm_ex(a, b, c, r, m, n, k, epi, 0, status, stream);
}

extern "C" TREE_API int tree_gemm_qkv(const void *a, const void *wqkv, void *q, void *k, void *v, int32_t m,
                                      int32_t nq, int32_t nkv, int32_t kdim, int32_t *status, tree_stream_t stream) {
  using namespace tree;
  if (!a || !wqkv || !q || !k || !v) return fail(TREE_ERR_INVALID_ARG, "tree_gemm_qkv: NULL argument");
  if (m < 0 || nq <= 0 || nkv <= 0 || kdim <= 0)
    return fail(TREE_ERR_INVALID_ARG, "tree_gemm_qkv: m %d, nq %d, nkv %d, k %d", m, nq, nkv, kdim);
  if (nq % 8 || nkv % 8 || kdim % 8)
    return fail(TREE_ERR_UNSUPPORTED, "tree_gemm_qkv: nq, nkv and k must be multiples of 8");
  if (!aligned16(a) || !aligned16(wqkv) || !aligned16(q) || !aligned16(k) || !aligned16(v))
    return fail(TREE_ERR_UNSUPPORTED, "tree_gemm_qkv: tensors must be 16-byte aligned");
  if (m == 0) return TREE_OK;
  const int n = nq + 2 * nkv;
  const cudaStream_t s = as_stream(stream);
  return narrow_tiles(m, TREE_GEMM_STORE)
             ? launch_gemm<64>(a, wqkv, q, nullptr, m, n, kdim, kEpiQKV, status, s, nq, nkv, k, v)
             : launch_gemm<256>(a, wqkv, q, nullptr, m, n, kdim, kEpiQKV, status, s, nq, nkv, k, v);
}
