// Helpers shared by the CUDA translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "internal.h"

namespace tree {

constexpr int kSMs = 152;  // GB300: 2 dies x 76 SMs

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

inline int launch_status(const char *what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return TREE_OK;
}

inline cudaStream_t as_stream(tree_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Number of SMs of the current device (cached per process; GB300 has 152).
int sm_count();

// Raise kernel `fn`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (device, kernel).
int set_max_dynamic_smem(const void *fn, int bytes, const char *who);

// 2-D TMA map over a row-major [rows, cols] f16 matrix: box_rows x 64-column
// boxes (128-byte rows), 128-byte swizzle, zero fill outside the matrix
// (box_rows 1: the map of tile::gather4 loads).  `who` names the caller in
// error messages.
int make_map(CUtensorMap *map, const void *base, int64_t cols, int64_t rows, const char *who, int box_rows = 128);

// Launch `kernel` on `s` allowed to start while the stream's previous kernel is
// still running (programmatic dependent launch): the kernel must execute
// griddepcontrol.wait before it reads anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Rotary embedding of 8 pairs (x_i, x_{i+d/2}): lo holds x_i .. x_{i+7}, hi the
// partners, cs their 8 {cos, sin} entries of the table.  The
// contraction into fma is written out, so that every kernel that rotates
// (tree_rope, and tree_attn_fwd rotating its query tiles) rounds alike.
__device__ __forceinline__ void rope_rotate8(uint4 &lo, uint4 &hi, const float4 (&cs)[4]) {
  __half2 *l = reinterpret_cast<__half2 *>(&lo);
  __half2 *h = reinterpret_cast<__half2 *>(&hi);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float4 c = cs[p];  // {cos_a, sin_a, cos_b, sin_b} for pairs 2p, 2p+1
    const float2 x1 = __half22float2(l[p]);
    const float2 x2 = __half22float2(h[p]);
    const float y1a = __fmaf_rn(x1.x, c.x, -__fmul_rn(x2.x, c.y));
    const float y2a = __fmaf_rn(x2.x, c.x, __fmul_rn(x1.x, c.y));
    const float y1b = __fmaf_rn(x1.y, c.z, -__fmul_rn(x2.y, c.w));
    const float y2b = __fmaf_rn(x2.y, c.z, __fmul_rn(x1.y, c.w));
    l[p] = __floats2half2_rn(y1a, y1b);
    h[p] = __floats2half2_rn(y2a, y2b);
  }
}

}  // namespace tree

namespace tree {
// The 8 {cos, sin} entries of pairs i0 .. i0+7 at position p of a [max_pos][d/2][2] table.
__device__ __forceinline__ void rope_table8(const float *cos_sin, int p, int d, int i0, float4 (&cs)[4]) {
  const float4 *t = reinterpret_cast<const float4 *>(cos_sin + ((size_t)p * (d / 2) + i0) * 2);
#pragma unroll
  for (int u = 0; u < 4; ++u) cs[u] = __ldg(t + u);
}
}  // namespace tree
