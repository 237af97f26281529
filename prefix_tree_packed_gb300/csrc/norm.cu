// tree_rmsnorm: the Llama RMSNorm before attention and before the MLP, over
// the packed tokens of a batch (basal-rs Architecture page, "01 / Request
// path: GPU forward pass": the Llama model in f16 over one compact token list).
//
//   y = f16( f16(x / sqrt(mean(x^2) + eps)) * w )
//
// One warp per row: a first pass sums the squares in f32 (8 values per lane
// and load), a second re-reads the row (now in L1) and writes y.  HBM-bound
// for many rows (x read once from memory, y written once); for a few rows the
// memory latency decides, so each pass issues its loads in chunks.

#include "common.cuh"
#include "sm103.cuh"
#include "tree_layer.h"

namespace tree {
namespace {

constexpr int kNormWarps = 8;
constexpr int kChunk = 8;   // 16-byte loads in flight per lane, first pass (x from memory)
constexpr int kChunk2 = 4;  // second pass (x again, now cached, and w): fewer registers

__global__ void __launch_bounds__(kNormWarps * 32) rmsnorm_kernel(const __half *x,
                                                                   const __half *__restrict__ w,
                                                                   __half *y, int rows, int cols,
                                                                   float eps) {
  sm103::griddep_wait();
  sm103::griddep_launch();
  const int row = blockIdx.x * kNormWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)row * cols);
  const int nv = cols / 8;
  // chunks of up to kChunk 16-byte loads per lane are issued together, so a row
  // costs one memory latency per chunk (two chunks at hidden 4096)
  float ss = 0.f;
  for (int i0 = 0; i0 < nv; i0 += 32 * kChunk) {
    uint4 v[kChunk];
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const int i = i0 + lane + 32 * u;
      v[u] = i < nv ? xr[i] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const __half2 *h = reinterpret_cast<const __half2 *>(&v[u]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(h[e]);
        ss = fmaf(f.x, f.x, ss);
        ss = fmaf(f.y, f.y, ss);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss / (float)cols + eps);
  const uint4 *wr = reinterpret_cast<const uint4 *>(w);
  uint4 *yr = reinterpret_cast<uint4 *>(y + (size_t)row * cols);
  // y may be x: each lane stores only elements it has already loaded
  for (int i0 = 0; i0 < nv; i0 += 32 * kChunk2) {
    uint4 v[kChunk2], wv[kChunk2];
#pragma unroll
    for (int u = 0; u < kChunk2; ++u) {
      const int i = i0 + lane + 32 * u;
      if (i < nv) {
        v[u] = xr[i];
        wv[u] = wr[i];
      }
    }
#pragma unroll
    for (int u = 0; u < kChunk2; ++u) {
      const int i = i0 + lane + 32 * u;
      if (i >= nv) continue;
      const __half2 *h = reinterpret_cast<const __half2 *>(&v[u]);
      const __half2 *hw = reinterpret_cast<const __half2 *>(&wv[u]);
      uint4 out;
      __half2 *ho = reinterpret_cast<__half2 *>(&out);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(h[e]);
        const __half2 n = __floats2half2_rn(f.x * inv, f.y * inv);
        ho[e] = __hmul2(n, hw[e]);
      }
      yr[i] = out;
    }
  }
}

}  // namespace
}  // namespace tree

extern "C" TREE_API int tree_rmsnorm(const void *x, const void *w, void *y, int32_t rows, int32_t cols, float eps,
                                     tree_stream_t stream) {
  using namespace tree;
  if (!x || !w || !y) return fail(TREE_ERR_INVALID_ARG, "tree_rmsnorm: NULL argument");
  if (rows < 0 || cols <= 0 || !(eps >= 0.f)) return fail(TREE_ERR_INVALID_ARG, "tree_rmsnorm: rows %d, cols %d", rows, cols);
  if (cols % 8 || cols > 16384) return fail(TREE_ERR_UNSUPPORTED, "tree_rmsnorm: cols %d (multiple of 8, <= 16384)", cols);
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return fail(TREE_ERR_UNSUPPORTED, "tree_rmsnorm: misaligned pointer");
  if (rows == 0) return TREE_OK;
  const int blocks = (rows + kNormWarps - 1) / kNormWarps;
  const cudaError_t e = launch_dependent(rmsnorm_kernel, dim3(blocks), dim3(kNormWarps * 32), 0, as_stream(stream),
                                         reinterpret_cast<const __half *>(x), reinterpret_cast<const __half *>(w),
                                         reinterpret_cast<__half *>(y), rows, cols, eps);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_rmsnorm: launch failed: %s", cudaGetErrorString(e));
  return launch_status("tree_rmsnorm");
}
