// tree_attn_fwd: attention over tree blocks for one forward chunk.
//
// A token sees the earlier tokens of its own block and every token of its
// ancestor blocks; sibling branches are masked, so each prompt's result equals
// computing it alone (basal-rs Architecture page, "03 / Packing: Attention
// over tree blocks").  With the planner's depth-first packing, key j is visible
// to query i iff j <= i < send[j].  Scores q.k * scale with scale = 1/sqrt(d)
// (AstrAI inference page, "KV Cache"); f16 storage, f32 softmax and
// accumulation ("01 / Request path: GPU forward pass").
//
// Work decomposition: one CTA per (query tile of 128 rows, q head), CTAs
// ordered longest tile first from the planner's per-chunk order.  The CTA walks
// the tile's list of 128-key tiles (empty tiles never appear in the list);
// full tiles skip the mask, partial tiles apply j <= i < send[j] per element.
// Online softmax in the log2 domain keeps one running max and sum per row.
//
// This file is the register-tile tensor-core version (mma.sync m16n8k16, f16
// in, f32 accumulate): 8 warps x 16 query rows, K/V/send tiles staged in
// shared memory with cp.async, XOR-swizzled 16-byte chunks for conflict-free
// ldmatrix.

#include <cmath>

#include "common.cuh"

namespace tree {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kWarps = 8;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// byte offset of 16-byte chunk c of row r in a swizzled tile with CH chunks per row
template <int CH>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * CH * 16 + ((c ^ (r & 7)) * 16));
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) attn_mma_kernel(
    const __half *__restrict__ q, const __half *__restrict__ k, const __half *__restrict__ v,
    __half *__restrict__ o, float *__restrict__ lse, const int32_t *__restrict__ send,
    const QTile *__restrict__ qtiles, const int32_t *__restrict__ ent, const int32_t *__restrict__ order,
    int32_t t0, int32_t q0, int32_t n_tot, int hq, int hkv, float scale_log2) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + BM * D * 2;
  uint8_t *sV = sK + BN * D * 2;
  int32_t *sSend = reinterpret_cast<int32_t *>(sV + BN * D * 2);

  const int h = blockIdx.x % hq;
  const int g = h / (hq / hkv);
  const QTile qt = qtiles[order[t0 + blockIdx.x / hq]];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- Q tile
  for (int x = tid; x < BM * CH; x += kWarps * 32) {
    const int r = x / CH, c = x % CH;
    const int row = qt.row0 + r;
    const bool ok = row < qt.row1;
    const __half *src = q + ((size_t)(ok ? row - q0 : 0) * hq + h) * D + c * 8;
    cp_async16(smem_u32(sQ) + swz<CH>(r, c), src, ok);
  }
  cp_async_commit();

  float acc[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const int qi0 = qt.row0 + warp * 16 + (lane >> 2);  // global query of c0/c1; +8 for c2/c3
  uint32_t qa[D / 16][4];

  for (int e = qt.ent0; e < qt.ent1; ++e) {
    const int code = ent[e];
    const int kt = code >> 1;
    const bool partial = code & 1;
    const int j0 = kt * BN;
    for (int x = tid; x < BN * CH; x += kWarps * 32) {
      const int r = x / CH, c = x % CH;
      const int key = j0 + r;
      const bool ok = key < n_tot;
      const size_t off = ((size_t)(ok ? key : 0) * hkv + g) * D + c * 8;
      cp_async16(smem_u32(sK) + swz<CH>(r, c), k + off, ok);
      cp_async16(smem_u32(sV) + swz<CH>(r, c), v + off, ok);
    }
    if (tid < BN / 4) cp_async16(smem_u32(sSend) + tid * 16, send + j0 + tid * 4, true);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    if (e == qt.ent0) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int r = warp * 16 + (lane & 15), c = kk * 2 + (lane >> 4);
        ldsm_x4(smem_u32(sQ) + swz<CH>(r, c), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
    }
    // ---- S = Q K^T for this warp's 16 rows x 128 keys
    float s[BN / 8][4];
#pragma unroll
    for (int n = 0; n < BN / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < BN / 16; ++np) {
        const int m = lane >> 3;
        const int r = np * 16 + (m >> 1) * 8 + (lane & 7), c = kk * 2 + (m & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(sK) + swz<CH>(r, c), b0, b1, b2, b3);
        mma16816(s[2 * np], qa[kk], b0, b1);
        mma16816(s[2 * np + 1], qa[kk], b2, b3);
      }
    }
    // ---- scale (log2 domain), mask, running max
    float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < BN / 8; ++n) {
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        float val = s[n][x] * scale_log2;
        if (partial) {
          const int jl = n * 8 + (lane & 3) * 2 + (x & 1);
          const int i = qi0 + (x >> 1) * 8;
          const int j = j0 + jl;
          if (!(j <= i && i < sSend[jl])) val = -INFINITY;
        }
        s[n][x] = val;
        mt[x >> 1] = fmaxf(mt[x >> 1], val);
      }
    }
    float alpha[2], mref[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mt[r] = fmaxf(mt[r], __shfl_xor_sync(0xffffffffu, mt[r], 1));
      mt[r] = fmaxf(mt[r], __shfl_xor_sync(0xffffffffu, mt[r], 2));
      const float mnew = fmaxf(mrow[r], mt[r]);
      mref[r] = mnew == -INFINITY ? 0.f : mnew;
      alpha[r] = ex2(mrow[r] - mref[r]);  // 0 when the old max is -inf
      mrow[r] = mnew;
      lrow[r] *= alpha[r];
    }
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      acc[j][0] *= alpha[0];
      acc[j][1] *= alpha[0];
      acc[j][2] *= alpha[1];
      acc[j][3] *= alpha[1];
    }
#pragma unroll
    for (int n = 0; n < BN / 8; ++n) {
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float p = ex2(s[n][x] - mref[x >> 1]);
        s[n][x] = p;
        lrow[x >> 1] += p;
      }
    }
    // ---- O += P V
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
      uint32_t a[4];
      a[0] = pack_half2(s[2 * kk][0], s[2 * kk][1]);
      a[1] = pack_half2(s[2 * kk][2], s[2 * kk][3]);
      a[2] = pack_half2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = pack_half2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int jp = 0; jp < D / 16; ++jp) {
        const int m = lane >> 3;
        const int r = kk * 16 + (m & 1) * 8 + (lane & 7), c = jp * 2 + (m >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(sV) + swz<CH>(r, c), b0, b1, b2, b3);
        mma16816(acc[2 * jp], a, b0, b1);
        mma16816(acc[2 * jp + 1], a, b2, b3);
      }
    }
    __syncthreads();
  }
  // ---- normalise and store
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = qi0 + r * 8;
    if (i >= qt.row1) continue;
    const float inv = 1.f / lrow[r];
    __half *dst = o + ((size_t)(i - q0) * hq + h) * D + (lane & 3) * 2;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      *reinterpret_cast<__half2 *>(dst + j * 8) =
          __floats2half2_rn(acc[j][2 * r] * inv, acc[j][2 * r + 1] * inv);
    }
    if (lse && (lane & 3) == 0) {
      const float mr = mrow[r] == -INFINITY ? 0.f : mrow[r];
      lse[(size_t)(i - q0) * hq + h] = (mr + log2f(lrow[r])) * 0.69314718055994531f;
    }
  }
}

template <int D>
int launch_mma(const Plan &P, const int32_t *img, int chunk, const void *q, const void *k, const void *v,
               void *o, float *lse, int hq, int hkv, float scale, cudaStream_t s) {
  const size_t smem = (size_t)(BM + 2 * BN) * D * 2 + BN * 4;
  auto kern = attn_mma_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_attn_fwd: %s", cudaGetErrorString(e));
  const int tiles = P.chunk_t1[chunk] - P.chunk_t0[chunk];
  const dim3 grid((unsigned)(tiles * hq));
  kern<<<grid, kWarps * 32, smem, s>>>(
      reinterpret_cast<const __half *>(q), reinterpret_cast<const __half *>(k),
      reinterpret_cast<const __half *>(v), reinterpret_cast<__half *>(o), lse, img + P.off_send,
      reinterpret_cast<const QTile *>(img + P.off_qtile), img + P.off_ent, img + P.off_order,
      P.chunk_t0[chunk], P.chunk_q0[chunk], P.n_tot, hq, hkv, scale * 1.4426950408889634f);
  return launch_status("tree_attn_fwd");
}

}  // namespace
}  // namespace tree

extern "C" TREE_API int tree_attn_fwd(const tree_plan_t *plan, const void *plan_dev, int32_t chunk,
                                      const void *q, const void *k, const void *v, void *o, float *lse,
                                      const tree_attn_params_t *params, int32_t *status, tree_stream_t stream) {
  using namespace tree;
  (void)status;
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
  if (d == 64) return launch_mma<64>(P, img, chunk, q, k, v, o, lse, hq, hkv, scale, s);
  return launch_mma<128>(P, img, chunk, q, k, v, o, lse, hq, hkv, scale, s);
}
