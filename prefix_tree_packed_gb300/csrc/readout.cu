// readout_decide: letter probabilities for both option orders, order 2 put back
// into the original option order, averaged and calibrated with the question
// type's temperature (basal-rs Architecture page, "02 / Basal protocol: Two
// option orders and calibration"):
//
//   p     = (softmax(l_order1) + reverse(softmax(l_order2))) / 2
//   p_cal = softmax(log(max(p, 1e-12)) / T)
//
// "reverse" maps order-2 letter k to original option n-1-k.  The decision is
// the argmax of p_cal (lowest index on ties); clamp, log, division by T > 0 and
// softmax are monotone and p sums to 1, so it is taken as the argmax of p.
// exp, log and the reciprocals use the hardware approximations (ex2.approx,
// lg2.approx, __fdividef): their error on these probabilities is ~1e-6, and
// the kernel is bound by its instruction count at large batches.
//
// Two work layouts.
//  * stride <= 32 (the usual 2-10 letters): a warp takes 32 consecutive
//    questions as one tile.  It gathers their logits rows flat (pass j, lane l
//    reads element l + 32 j of the 32 x stride tile), so one load instruction
//    touches a few neighbouring rows rather than 32 scattered ones; the rows go
//    to shared memory at an odd pitch, the order-2 row already reversed into
//    original option order; each lane then decides one question in registers
//    with straight-line code, and the warp writes the tile's p_cal (and p_avg)
//    rows back as one contiguous, coalesced span.  Strides 1..16 have one
//    instance each (all tile addressing is compile-time).
//  * stride > 32 (up to 255 letters): one warp per question, lane l holding
//    letters l, l + 32, ..., reductions by shuffles.

#include <cfloat>

#include "common.cuh"
#include "sm103.cuh"

namespace tree {
namespace {

constexpr float kClamp = 1e-12f;

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// K = letters per lane (G * K >= largest stride handled).
template <int G, int K>
__global__ void __launch_bounds__(256) readout_kernel(const float *__restrict__ logits, int stride,
                                                      const int32_t *__restrict__ r1,
                                                      const int32_t *__restrict__ r2,
                                                      const int32_t *__restrict__ nl,
                                                      const float *__restrict__ temp, int nq,
                                                      float *__restrict__ p_cal,
                                                      float *__restrict__ p_avg,
                                                      int32_t *__restrict__ choice,
                                                      int32_t *__restrict__ status) {
  sm103::griddep_wait();    // the logits may come from the kernel before this one in the stream
  sm103::griddep_launch();  // the next kernel may launch (it waits for this one if it reads its results)
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const int q = gtid / G;
  const int lane = gtid % G;
  // whole groups leave together, so shuffles below see full groups
  if (q >= nq) return;
  const int n = nl[q];
  const float T = temp[q];
  const bool bad = n < 1 || n > stride || n > 255 || !(T > 0.f);
  float *pc_row = p_cal + (size_t)q * stride;
  float *pa_row = p_avg ? p_avg + (size_t)q * stride : nullptr;
  if (bad) {
    for (int i = lane; i < stride; i += G) {
      pc_row[i] = 0.f;
      if (pa_row) pa_row[i] = 0.f;
    }
    if (lane == 0) {
      if (choice) choice[q] = -1;
      if (status) atomicExch(status, TREE_ERR_INVALID_ARG);
    }
    return;
  }
  const float *a = logits + (size_t)r1[q] * stride;
  const float *b = logits + (size_t)r2[q] * stride;
  float x1[K], x2[K];
  float m1 = -FLT_MAX, m2 = -FLT_MAX;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int i = lane + G * k;
    if (i < n) {
      x1[k] = a[i];
      x2[k] = b[n - 1 - i];  // order-2 letter of original option i
      m1 = fmaxf(m1, x1[k]);
      m2 = fmaxf(m2, x2[k]);
    }
  }
  m1 = group_max<G>(m1);
  m2 = group_max<G>(m2);
  float s1 = 0.f, s2 = 0.f;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if (lane + G * k < n) {
      x1[k] = __expf(x1[k] - m1);
      x2[k] = __expf(x2[k] - m2);
      s1 += x1[k];
      s2 += x2[k];
    }
  }
  s1 = group_sum<G>(s1);
  s2 = group_sum<G>(s2);
  const float inv1 = __fdividef(1.f, s1), inv2 = __fdividef(1.f, s2), invT = __fdividef(1.f, T);
  // p (kept in x1), its calibrated logit (kept in x2), argmax of p
  float m3 = -FLT_MAX, best = -1.f;
  int arg = 0x7fffffff;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int i = lane + G * k;
    if (i < n) {
      const float p = 0.5f * (x1[k] * inv1 + x2[k] * inv2);
      x1[k] = p;
      x2[k] = __logf(fmaxf(p, kClamp)) * invT;
      m3 = fmaxf(m3, x2[k]);
      if (p > best) {  // letters visited in increasing index: first maximum wins
        best = p;
        arg = i;
      }
    }
  }
  m3 = group_max<G>(m3);
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oa = __shfl_xor_sync(0xffffffffu, arg, o);
    if (ob > best || (ob == best && oa < arg)) {
      best = ob;
      arg = oa;
    }
  }
  float s3 = 0.f;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if (lane + G * k < n) {
      x2[k] = __expf(x2[k] - m3);
      s3 += x2[k];
    }
  }
  s3 = group_sum<G>(s3);
  const float inv3 = __fdividef(1.f, s3);
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int i = lane + G * k;
    if (i < n) {
      pc_row[i] = x2[k] * inv3;
      if (pa_row) pa_row[i] = x1[k];
    }
  }
  for (int i = n + lane; i < stride; i += G) {
    pc_row[i] = 0.f;
    if (pa_row) pa_row[i] = 0.f;
  }
  if (lane == 0 && choice) choice[q] = arg;
}

constexpr int kTileWarps = 4;  // warps (32-question tiles) per block
constexpr float kLog2e = 1.4426950408889634f;

// Tile layout, stride <= K <= 32.  A warp takes 32 consecutive questions.
// Shared memory per warp: two 32-row input tiles (order 1, order 2) at pitch
// `pitch` = stride rounded up to odd, so that lane l reading row l, column k
// hits bank (l * pitch + k) mod 32: all distinct; after the decision the same
// space holds the tile's p_cal and p_avg rows at pitch `stride`, i.e. exactly
// as they lie in global memory.  A second area holds each question's
// {r1, r2, n} for the gather.  EXACT: stride == K, known at compile time (all
// addressing constant-folds); otherwise stride is the runtime `stride_rt` <= K
// and `magic` = ceil(2^16 / stride): for e < 32 * 32, (e * magic) >> 16 is
// exactly e / stride (the rounding error e / 2^16 < 1/64 stays below the gap
// 1/stride between e / stride and the next integer).  V = 2 (even strides,
// 8-byte aligned logits): the gather moves letter pairs.
//
// The order-2 row is reversed while it is gathered (slot i of a question with
// n letters takes its letter n-1-i, the one that names original option i), and the
// slots past n hold -inf, so each lane decides its question with the same
// straight-line code over all K slots: exp(-inf) = 0 makes the padding vanish
// from both softmax sums and gives it p = 0; only the calibrated logit needs
// the explicit k < n test (log of the clamp is finite).
template <int K, bool EXACT, int V>
__global__ void __launch_bounds__(kTileWarps * 32) readout_tile_kernel(
    const float *__restrict__ logits, int stride_rt, uint32_t magic, const int32_t *__restrict__ r1,
    const int32_t *__restrict__ r2, const int32_t *__restrict__ nl, const float *__restrict__ temp, int nq,
    float *__restrict__ p_cal, float *__restrict__ p_avg, int32_t *__restrict__ choice,
    int32_t *__restrict__ status, int vec_out) {
  static_assert(V == 1 || (V == 2 && EXACT && K % 2 == 0), "letter pairs need an even, compile-time stride");
  extern __shared__ float tile_smem[];
  const int S = EXACT ? K : stride_rt;
  const int pitch = S | 1;
  constexpr int NP = EXACT ? K / V : K;  // gather passes (runtime stride: the first S of K)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t q0 = ((int64_t)blockIdx.x * kTileWarps + warp) * 32;
  if (q0 >= nq) return;  // whole warps leave together
  const int nv = (int)min((int64_t)32, (int64_t)nq - q0);
  float *sa = tile_smem + (size_t)warp * 64 * pitch;
  float *sb = sa + 32 * pitch;
  int4 *meta = reinterpret_cast<int4 *>(tile_smem + (size_t)kTileWarps * 64 * pitch) + warp * 32;
  // group g (V letters) of the tile's flat 32 x S span -> its question
  auto row_of = [&](int g) -> int {
    return EXACT ? (int)((uint32_t)g / (uint32_t)(K / V)) : (int)(((uint32_t)g * magic) >> 16);
  };

  // The question records are read before waiting for the kernel ahead in the
  // stream (only the logits come from it), so their memory latency overlaps
  // that kernel's tail; a caller's kernel that lets dependents launch early must
  // not write them (the library's kernels never do).
  int my_n = 0;
  float T = 1.f;
  int4 m = make_int4(0, 0, 0, 0);
  if (lane < nv) {
    m.x = r1[q0 + lane];
    m.y = r2[q0 + lane];
    my_n = nl[q0 + lane];
    T = temp[q0 + lane];
  }
  sm103::griddep_wait();    // the logits may come from the kernel before this one in the stream
  sm103::griddep_launch();  // the next kernel may launch (it waits for this one if it reads its results)
  const bool bad = lane < nv && (my_n < 1 || my_n > S || my_n > 255 || !(T > 0.f));
  m.z = (lane < nv && !bad) ? my_n : 0;  // letters to load
  meta[lane] = m;
  __syncwarp();

  // gather: pass j, lane l takes group l + 32 j of the flat span, so one load
  // instruction touches a few neighbouring rows; all loads are in flight
  // before the first shared-memory store.  Slot s of the order-2 row takes
  // letter n-1-s of its logits row (read backwards from global memory).
  float va[NP * V], vb[NP * V];
  int off[NP];
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    const int g = lane + 32 * j;
    const int qq = row_of(g) & 31;  // < 32 whenever j < S / V
    const int i = (g - qq * (S / V)) * V;
    const int4 mq = meta[qq];
    const int nn = mq.z;
    off[j] = qq * pitch + i;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      va[j * V + v] = -INFINITY;
      vb[j * V + v] = -INFINITY;
    }
    if ((EXACT || j < S) && i < nn) {
      const float *rowb = logits + (size_t)mq.y * S + (nn - 1 - i);  // slot i + v: rowb[-v]
      if (V == 2) {
        const float2 a2 = *reinterpret_cast<const float2 *>(logits + (size_t)mq.x * S + i);
        va[j * V] = a2.x;
        vb[j * V] = rowb[0];
        if (i + 1 < nn) {
          va[j * V + V - 1] = a2.y;
          vb[j * V + V - 1] = rowb[-1];
        }
      } else {
        va[j * V] = logits[(size_t)mq.x * S + i];
        vb[j * V] = rowb[0];
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    if (EXACT || j < S) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        sa[off[j] + v] = va[j * V + v];
        sb[off[j] + v] = vb[j * V + v];
      }
    }
  }
  __syncwarp();

  // decide: lane = question, its two rows in registers (lanes past nv and bad
  // questions compute on whatever their rows hold; their results are not kept)
  float x1[K], x2[K];
  {
    const float *ra_s = sa + lane * pitch, *rb_s = sb + lane * pitch;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      x1[k] = (EXACT || k < S) ? ra_s[k] : -INFINITY;
      x2[k] = (EXACT || k < S) ? rb_s[k] : -INFINITY;
    }
  }
  __syncwarp();  // every row is in registers: the space now takes the outputs
  float m1 = -FLT_MAX, m2 = -FLT_MAX;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    m1 = fmaxf(m1, x1[k]);
    m2 = fmaxf(m2, x2[k]);
  }
  // exp(x - m) as 2^(x log2 e - m log2 e)
  const float c1 = m1 * kLog2e, c2 = m2 * kLog2e;
  float s1 = 0.f, s2 = 0.f;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    x1[k] = sm103::ex2(fmaf(x1[k], kLog2e, -c1));
    x2[k] = sm103::ex2(fmaf(x2[k], kLog2e, -c2));
    s1 += x1[k];
    s2 += x2[k];
  }
  const float h1 = 0.5f * __fdividef(1.f, s1), h2 = 0.5f * __fdividef(1.f, s2);
  const float invT = __fdividef(1.f, T);
  // p, and its calibrated logit in base 2: ln(p) / T = log2(p) / T * ln 2, and
  // the softmax of z is the base-2 softmax of z log2 e, so the ln 2 and log2 e
  // cancel
  float m3 = -FLT_MAX, best = -1.f;
  int arg = 0;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const float p = fmaf(x1[k], h1, x2[k] * h2);
    x1[k] = p;
    x2[k] = k < my_n ? sm103::lg2(fmaxf(p, kClamp)) * invT : -INFINITY;
    m3 = fmaxf(m3, x2[k]);
    if (p > best) {  // increasing index: the first maximum wins; padding has p = 0
      best = p;
      arg = k;
    }
  }
  float s3 = 0.f;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    x2[k] = sm103::ex2(x2[k] - m3);
    s3 += x2[k];
  }
  const float inv3 = __fdividef(1.f, s3);
  {
    // a bad question's rows are zero (its arithmetic ran on -inf rows: NaN)
    float *pc_s = sa + lane * S, *pa_s = sb + lane * S;
#pragma unroll
    for (int k = 0; k < K; ++k)
      if (EXACT || k < S) {
        pc_s[k] = bad ? 0.f : x2[k] * inv3;
        pa_s[k] = bad ? 0.f : x1[k];
      }
  }
  if (lane < nv) {
    if (choice) choice[q0 + lane] = bad ? -1 : arg;
    if (bad && status) atomicExch(status, TREE_ERR_INVALID_ARG);
  }
  __syncwarp();

  // write back: the tile's rows are one contiguous span of nv * S floats,
  // staged in the same order
  float *pc = p_cal + q0 * S;
  float *pa = p_avg ? p_avg + q0 * S : nullptr;
  const int span = nv * S;
  int e0 = 0;
  if (vec_out) {  // p_cal and p_avg 16-byte aligned (the tile start is: q0 * S * 4 is a multiple of 128)
    const int n4 = span >> 2;
    if (EXACT) {  // at most 8 K float4 per tile: a fixed number of passes
#pragma unroll
      for (int t = 0; t < (8 * K + 31) / 32; ++t) {
        const int e = lane + 32 * t;
        if (e < n4) {
          reinterpret_cast<float4 *>(pc)[e] = reinterpret_cast<const float4 *>(sa)[e];
          if (pa) reinterpret_cast<float4 *>(pa)[e] = reinterpret_cast<const float4 *>(sb)[e];
        }
      }
    } else {
      for (int e = lane; e < n4; e += 32) {
        reinterpret_cast<float4 *>(pc)[e] = reinterpret_cast<const float4 *>(sa)[e];
        if (pa) reinterpret_cast<float4 *>(pa)[e] = reinterpret_cast<const float4 *>(sb)[e];
      }
    }
    e0 = n4 << 2;
  }
  for (int e = e0 + lane; e < span; e += 32) {
    pc[e] = sa[e];
    if (pa) pa[e] = sb[e];
  }
}

// strides 1..16 (the usual letter counts) each get their own instance; even
// strides also one that gathers letter pairs
using TileKernel = void (*)(const float *, int, uint32_t, const int32_t *, const int32_t *, const int32_t *,
                            const float *, int, float *, float *, int32_t *, int32_t *, int);
constexpr int kExactStrides = 16;
const TileKernel kExactTile[kExactStrides] = {
    readout_tile_kernel<1, true, 1>,  readout_tile_kernel<2, true, 1>,  readout_tile_kernel<3, true, 1>,
    readout_tile_kernel<4, true, 1>,  readout_tile_kernel<5, true, 1>,  readout_tile_kernel<6, true, 1>,
    readout_tile_kernel<7, true, 1>,  readout_tile_kernel<8, true, 1>,  readout_tile_kernel<9, true, 1>,
    readout_tile_kernel<10, true, 1>, readout_tile_kernel<11, true, 1>, readout_tile_kernel<12, true, 1>,
    readout_tile_kernel<13, true, 1>, readout_tile_kernel<14, true, 1>, readout_tile_kernel<15, true, 1>,
    readout_tile_kernel<16, true, 1>};
const TileKernel kPairTile[kExactStrides / 2] = {
    readout_tile_kernel<2, true, 2>,  readout_tile_kernel<4, true, 2>,  readout_tile_kernel<6, true, 2>,
    readout_tile_kernel<8, true, 2>,  readout_tile_kernel<10, true, 2>, readout_tile_kernel<12, true, 2>,
    readout_tile_kernel<14, true, 2>, readout_tile_kernel<16, true, 2>};

}  // namespace
}  // namespace tree

extern "C" TREE_API int readout_decide(const float *logits, int32_t stride, const int32_t *r1,
                                       const int32_t *r2, const int32_t *n_letters,
                                       const float *temperature, int32_t n_q, float *p_cal,
                                       float *p_avg, int32_t *choice, int32_t *status,
                                       tree_stream_t stream) {
  using namespace tree;
  if (n_q < 0 || stride <= 0) return fail(TREE_ERR_INVALID_ARG, "readout_decide: n_q %d, stride %d", n_q, stride);
  if (n_q == 0) return TREE_OK;
  if (!logits || !r1 || !r2 || !n_letters || !temperature || !p_cal)
    return fail(TREE_ERR_INVALID_ARG, "readout_decide: NULL argument");
  const cudaStream_t s = as_stream(stream);
  if (stride <= 32) {
    const int pitch = stride | 1;
    const uint32_t magic = (65536u + (uint32_t)stride - 1u) / (uint32_t)stride;
    const int64_t warps = ((int64_t)n_q + 31) / 32;
    const int blocks = (int)((warps + kTileWarps - 1) / kTileWarps);
    const size_t smem = ((size_t)kTileWarps * 64 * pitch + (size_t)kTileWarps * 32 * 4) * sizeof(float);
    const bool pairs = stride % 2 == 0 && reinterpret_cast<uintptr_t>(logits) % 8 == 0;
    const int vec_out = reinterpret_cast<uintptr_t>(p_cal) % 16 == 0 && reinterpret_cast<uintptr_t>(p_avg) % 16 == 0;
    const TileKernel kern = stride > kExactStrides ? readout_tile_kernel<32, false, 1>
                            : pairs               ? kPairTile[stride / 2 - 1]
                                                  : kExactTile[stride - 1];
    // launched to overlap the previous kernel's tail; the kernels wait for it before reading
    const cudaError_t e = launch_dependent(kern, dim3(blocks), dim3(kTileWarps * 32), smem, s, logits, stride, magic,
                                           r1, r2, n_letters, temperature, n_q, p_cal, p_avg, choice, status, vec_out);
    if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "readout_decide: launch failed: %s", cudaGetErrorString(e));
  } else {
    const int threads = 256;
    const int64_t lanes = (int64_t)n_q * 32;
    const int blocks = (int)((lanes + threads - 1) / threads);
    const cudaError_t e = launch_dependent(readout_kernel<32, 8>, dim3(blocks), dim3(threads), 0, s, logits, stride,
                                           r1, r2, n_letters, temperature, n_q, p_cal, p_avg, choice, status);
    if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "readout_decide: launch failed: %s", cudaGetErrorString(e));
  }
  return launch_status("readout_decide");
}
