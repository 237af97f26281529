// tree_rope: rotary embedding at tree positions, in place on Q and K.
//
// The rotary position of a token is its position in its own prompt (basal-rs
// Architecture page, "03 / Packing: Attention over tree blocks"); the planner's
// pos table holds it.  Pairs (i, i + d/2) are rotated by pos * theta^(-2i/d)
// (the Llama "rotate half" layout):
//
//   y_i       = x_i cos - x_{i+d/2} sin
//   y_{i+d/2} = x_{i+d/2} cos + x_i sin
//
// cos/sin come from an f32 table [max_pos][d/2][2] that the host fills in
// double precision (tree_rope_table), the table form of the AstrAI inference
// page ("Rotary Embedding Backend"); evaluating pos * inv_freq in f32 instead
// would put ~2e-3 rad of error on the angle at position 32k.
//
// The kernel is a streaming pass over the chunk's Q rows and K rows: one
// thread rotates 8 pairs of one head (two 16-byte loads and stores) of one
// token row; threads of a warp cover consecutive pairs and heads of a row, so
// every access is a full 32-byte sector; the cos/sin table stays in L1/L2.
// The pass is bound by memory latency, so it is written for occupancy: one row
// per thread keeps it at 32 registers and many small blocks in flight
// (measured on GB300 against 2, 3 and 4 rows per thread, a register cap, and a
// bulk-copy pipeline through shared memory, all slower).

#include <cmath>

#include "common.cuh"
#include "sm103.cuh"

namespace tree {
namespace {

using namespace sm103;

constexpr int kRopeMaxThreads = 512;
constexpr int kRopeRows = 1;  // token rows per block

// Block (x, y): token rows [kRopeRows * x, +kRopeRows) of the chunk, items
// [blockDim.x * y, +blockDim.x) of a row, where a row's items are (q heads, then kv
// heads) x (d/16 groups of 8 pairs).  A thread keeps the same item for all its
// rows, so the index arithmetic is done once.
__global__ void __launch_bounds__(kRopeMaxThreads) rope_kernel(__half *__restrict__ q, __half *__restrict__ k,
                                                            const int32_t *__restrict__ pos, int32_t q0,
                                                            int32_t nrows, int hq, int hkv, int d,
                                                            const float *__restrict__ cos_sin, int32_t max_pos) {
  // launched to overlap the kernel before it in the stream: wait for it before
  // reading the positions or the rows (it may write them), then let the next
  // kernel launch (it waits for this grid before reading)
  griddep_wait();
  griddep_launch();
  const int per_head = d / 16;
  const int item = blockIdx.y * blockDim.x + threadIdx.x;
  if (item >= (hq + hkv) * per_head) return;
  const int head = item / per_head;
  const int c = item - head * per_head;
  const bool is_q = head < hq;
  __half *base = is_q ? q + (size_t)head * d + 8 * c : k + (size_t)(head - hq) * d + 8 * c;
  const size_t row_stride = (size_t)(is_q ? hq : hkv) * d;
  const int r0 = blockIdx.x * kRopeRows;
  uint4 lo[kRopeRows], hi[kRopeRows];
  int p[kRopeRows];
  __half *x[kRopeRows];
#pragma unroll
  for (int u = 0; u < kRopeRows; ++u) {
    const int r = r0 + u;
    p[u] = -1;
    if (r < nrows) {
      p[u] = __ldg(pos + q0 + r);
      x[u] = base + (size_t)(is_q ? r : q0 + r) * row_stride;
      lo[u] = *reinterpret_cast<const uint4 *>(x[u]);
      hi[u] = *reinterpret_cast<const uint4 *>(x[u] + d / 2);
    }
  }
#pragma unroll
  for (int u = 0; u < kRopeRows; ++u) {
    // a position outside the table cannot come from a plan the host checked
    if (p[u] < 0 || p[u] >= max_pos) continue;
    float4 cs[4];
    rope_table8(cos_sin, p[u], d, 8 * c, cs);
    rope_rotate8(lo[u], hi[u], cs);
    *reinterpret_cast<uint4 *>(x[u]) = lo[u];
    *reinterpret_cast<uint4 *>(x[u] + d / 2) = hi[u];
  }
}

}  // namespace
}  // namespace tree

extern "C" TREE_API int tree_rope_table(float *host_out, int32_t max_pos, int32_t d, double theta) {
  using namespace tree;
  if (!host_out || max_pos <= 0 || d <= 0 || d % 2 || !(theta > 0))
    return fail(TREE_ERR_INVALID_ARG, "tree_rope_table: max_pos %d, d %d, theta %g", max_pos, d, theta);
  const int h = d / 2;
  for (int32_t p = 0; p < max_pos; ++p)
    for (int i = 0; i < h; ++i) {
      const double a = (double)p * std::pow(theta, -2.0 * i / d);
      host_out[((size_t)p * h + i) * 2 + 0] = (float)std::cos(a);
      host_out[((size_t)p * h + i) * 2 + 1] = (float)std::sin(a);
    }
  return TREE_OK;
}

extern "C" TREE_API int tree_rope(const tree_plan_t *plan, const void *plan_dev, int32_t chunk, void *q,
                                  void *k, int32_t hq, int32_t hkv, int32_t d, const float *cos_sin,
                                  int32_t max_pos, int32_t *status, tree_stream_t stream) {
  using namespace tree;
  (void)status;  // the kernel never waits, so it has nothing to report
  if (!plan || !plan_dev || !k || !cos_sin) return fail(TREE_ERR_INVALID_ARG, "tree_rope: NULL argument");
  if (!q) hq = 0;  // keys only
  const Plan &P = plan->p;
  if (chunk < 0 || chunk >= P.n_chunks) return fail(TREE_ERR_INVALID_ARG, "tree_rope: chunk %d out of range", chunk);
  if (hq < 0 || (q && hq == 0) || hkv <= 0 || d <= 0 || d % 16 || d > 256)
    return fail(TREE_ERR_UNSUPPORTED, "tree_rope: hq %d hkv %d d %d (d must be a multiple of 16, <= 256)", hq,
                hkv, d);
  if (max_pos < P.max_pos)
    return fail(TREE_ERR_INVALID_ARG, "tree_rope: table has %d positions, plan needs %d", max_pos, P.max_pos);
  if ((q && !aligned16(q)) || !aligned16(k) || !aligned16(cos_sin) || !aligned16(plan_dev))
    return fail(TREE_ERR_UNSUPPORTED, "tree_rope: pointers must be 16-byte aligned");
  const int32_t q0 = P.chunk_q0[chunk], n = P.chunk_q1[chunk] - q0;
  const int items = (hq + hkv) * (d / 16);
  const int threads = std::min(kRopeMaxThreads, (items + 31) / 32 * 32);
  const dim3 grid((unsigned)((n + kRopeRows - 1) / kRopeRows), (unsigned)((items + threads - 1) / threads));
  const int32_t *pos = reinterpret_cast<const int32_t *>(plan_dev) + P.off_pos;
  const cudaError_t e = launch_dependent(rope_kernel, grid, dim3(threads), 0, as_stream(stream),
                                         reinterpret_cast<__half *>(q), reinterpret_cast<__half *>(k), pos, q0, n, hq,
                                         hkv, d, cos_sin, max_pos);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_rope: launch failed: %s", cudaGetErrorString(e));
  return launch_status("tree_rope");
}
