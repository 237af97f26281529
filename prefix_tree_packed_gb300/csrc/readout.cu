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
// exp, log and the reciprocals use the hardware approximations (__expf,
// __logf, __fdividef): their error on these probabilities is ~1e-6, and the
// kernel is bound by its instruction count at large batches.
//
// Two work layouts.
//  * stride <= 32 (the usual 2-10 letters): a warp takes 32 consecutive
//    questions as one tile.  It gathers their logits rows flat (pass j, lane l
//    reads element l + 32 j of the 32 x stride tile), so one load instruction
//    touches a few neighbouring rows rather than 32 scattered ones; the rows go
//    to shared memory at an odd pitch, each lane decides one question from
//    there without bank conflicts, and the warp writes the tile's p_cal (and
//    p_avg) rows back as one contiguous, coalesced span.
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

// Decision for one question held in lane registers: x1 = order-1 logits, x2 =
// order-2 logits already put into original option order, n letters (1..K).
// Leaves p_avg in x1 and p_cal in x2; returns the argmax of p.
template <int K>
__device__ __forceinline__ int decide_lane(float (&x1)[K], float (&x2)[K], int n, float T) {
  float m1 = -FLT_MAX, m2 = -FLT_MAX;
#pragma unroll
  for (int k = 0; k < K; ++k)
    if (k < n) {
      m1 = fmaxf(m1, x1[k]);
      m2 = fmaxf(m2, x2[k]);
    }
  float s1 = 0.f, s2 = 0.f;
#pragma unroll
  for (int k = 0; k < K; ++k)
    if (k < n) {
      x1[k] = __expf(x1[k] - m1);
      x2[k] = __expf(x2[k] - m2);
      s1 += x1[k];
      s2 += x2[k];
    }
  const float inv1 = __fdividef(1.f, s1), inv2 = __fdividef(1.f, s2), invT = __fdividef(1.f, T);
  float m3 = -FLT_MAX, best = -1.f;
  int arg = 0;
#pragma unroll
  for (int k = 0; k < K; ++k)
    if (k < n) {
      const float p = 0.5f * (x1[k] * inv1 + x2[k] * inv2);
      x1[k] = p;
      x2[k] = __logf(fmaxf(p, kClamp)) * invT;
      m3 = fmaxf(m3, x2[k]);
      if (p > best) {  // increasing index: the first maximum wins
        best = p;
        arg = k;
      }
    }
  float s3 = 0.f;
#pragma unroll
  for (int k = 0; k < K; ++k)
    if (k < n) {
      x2[k] = __expf(x2[k] - m3);
      s3 += x2[k];
    }
  const float inv3 = __fdividef(1.f, s3);
#pragma unroll
  for (int k = 0; k < K; ++k)
    if (k < n) x2[k] *= inv3;
  return arg;
}

constexpr int kTileWarps = 4;  // warps (32-question tiles) per block
constexpr int kLoopQuestions = 262144;  // from this batch size on, decide with loops (measured crossover)

// Tile layout, stride <= K <= 32.  Shared memory per warp: two 32-row tiles
// (order 1, order 2) at pitch `pitch` = stride rounded up to odd.  `magic` =
// ceil(2^16 / stride): for e < 32 * 32 and stride <= 32, (e * magic) >> 16 is
// exactly e / stride (the rounding error e / 2^16 < 1/64 stays below the gap
// 1/stride between e / stride and the next integer).
template <int K, bool LOOPS>
__global__ void __launch_bounds__(kTileWarps * 32) readout_tile_kernel(
    const float *__restrict__ logits, int stride, int pitch, uint32_t magic, const int32_t *__restrict__ r1,
    const int32_t *__restrict__ r2, const int32_t *__restrict__ nl, const float *__restrict__ temp, int nq,
    float *__restrict__ p_cal, float *__restrict__ p_avg, int32_t *__restrict__ choice,
    int32_t *__restrict__ status) {
  extern __shared__ float tile_smem[];
  sm103::griddep_wait();    // the logits may come from the kernel before this one in the stream
  sm103::griddep_launch();  // the next kernel may launch (it waits for this one if it reads its results)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t q0 = ((int64_t)blockIdx.x * kTileWarps + warp) * 32;
  if (q0 >= nq) return;  // whole warps leave together
  const int nv = (int)min((int64_t)32, (int64_t)nq - q0);
  float *sa = tile_smem + (size_t)warp * 64 * pitch;
  float *sb = sa + 32 * pitch;

  int my_r1 = 0, my_r2 = 0, my_n = 0;
  float T = 1.f;
  if (lane < nv) {
    my_r1 = r1[q0 + lane];
    my_r2 = r2[q0 + lane];
    my_n = nl[q0 + lane];
    T = temp[q0 + lane];
  }
  const bool bad = lane < nv && (my_n < 1 || my_n > stride || my_n > 255 || !(T > 0.f));
  const int n_load = (lane < nv && !bad) ? my_n : 0;

  // gather: all loads in flight before the shared-memory stores
  float va[K], vb[K];
#pragma unroll
  for (int j = 0; j < K; ++j) {
    const int e = lane + 32 * j;
    const int qq = (int)(((uint32_t)e * magic) >> 16);
    const int i = e - qq * stride;
    // qq < 32 whenever j < stride; shuffles run on every lane with in-range sources
    const int src = qq & 31;
    const int ra = __shfl_sync(0xffffffffu, my_r1, src);
    const int rb = __shfl_sync(0xffffffffu, my_r2, src);
    const int nn = __shfl_sync(0xffffffffu, n_load, src);
    va[j] = 0.f;
    vb[j] = 0.f;
    if (j < stride && i < nn) {
      va[j] = logits[(size_t)ra * stride + i];
      vb[j] = logits[(size_t)rb * stride + i];
    }
  }
#pragma unroll
  for (int j = 0; j < K; ++j) {
    const int e = lane + 32 * j;
    if (j < stride) {
      const int qq = (int)(((uint32_t)e * magic) >> 16);
      const int i = e - qq * stride;
      sa[qq * pitch + i] = va[j];
      sb[qq * pitch + i] = vb[j];
    }
  }
  __syncwarp();

  // decide: lane = question; each lane touches only its own two rows.  Small
  // batches keep the letters in registers (fully unrolled: shortest latency);
  // large ones decide from the rows in shared memory with loops over the n
  // letters (fewer registers and instructions: more warps in flight).  Both
  // forms do the same operations in the same order.
  if (!LOOPS) {
  if (lane < nv) {
    float *ra_s = sa + lane * pitch, *rb_s = sb + lane * pitch;
    if (bad) {
      for (int i = 0; i < stride; ++i) ra_s[i] = rb_s[i] = 0.f;
      if (choice) choice[q0 + lane] = -1;
      if (status) atomicExch(status, TREE_ERR_INVALID_ARG);
    } else {
      float x1[K], x2[K];
#pragma unroll
      for (int k = 0; k < K; ++k)
        if (k < my_n) {
          x1[k] = ra_s[k];
          x2[k] = rb_s[my_n - 1 - k];  // order-2 letter of original option k
        }
      const int arg = decide_lane<K>(x1, x2, my_n, T);
#pragma unroll
      for (int k = 0; k < K; ++k)
        if (k < stride) {
          ra_s[k] = k < my_n ? x2[k] : 0.f;
          rb_s[k] = k < my_n ? x1[k] : 0.f;
        }
      if (choice) choice[q0 + lane] = arg;
    }
  }
  } else {
  if (lane < nv) {
    float *ra_s = sa + lane * pitch, *rb_s = sb + lane * pitch;
    if (bad) {
      for (int i = 0; i < stride; ++i) ra_s[i] = rb_s[i] = 0.f;
      if (choice) choice[q0 + lane] = -1;
      if (status) atomicExch(status, TREE_ERR_INVALID_ARG);
    } else {
      const int n = my_n;
      float m1 = -FLT_MAX, m2 = -FLT_MAX;
      for (int i = 0; i < n; ++i) {
        m1 = fmaxf(m1, ra_s[i]);
        m2 = fmaxf(m2, rb_s[i]);
      }
      float s1 = 0.f, s2 = 0.f;
      // option i of order 2 is letter n-1-i of its row; each slot is read, then overwritten
      for (int i = 0; i < n; ++i) {
        const float e1 = __expf(ra_s[i] - m1), e2 = __expf(rb_s[n - 1 - i] - m2);
        s1 += e1;
        s2 += e2;
        ra_s[i] = e1;
        rb_s[n - 1 - i] = e2;
      }
      const float inv1 = __fdividef(1.f, s1), inv2 = __fdividef(1.f, s2), invT = __fdividef(1.f, T);
      float m3 = -FLT_MAX, best = -1.f;
      int arg = 0;
      for (int i = 0; i < n; ++i) {
        const float p = 0.5f * (ra_s[i] * inv1 + rb_s[n - 1 - i] * inv2);
        const float lg = __logf(fmaxf(p, kClamp)) * invT;
        ra_s[i] = lg;
        rb_s[n - 1 - i] = p;  // in reversed order for now
        m3 = fmaxf(m3, lg);
        if (p > best) {  // increasing index: the first maximum wins
          best = p;
          arg = i;
        }
      }
      for (int i = 0; i < n / 2; ++i) {  // p_avg into original option order
        const float t = rb_s[i];
        rb_s[i] = rb_s[n - 1 - i];
        rb_s[n - 1 - i] = t;
      }
      for (int i = n; i < stride; ++i) rb_s[i] = 0.f;
      float s3 = 0.f;
      for (int i = 0; i < n; ++i) {
        const float e3 = __expf(ra_s[i] - m3);
        s3 += e3;
        ra_s[i] = e3;
      }
      const float inv3 = __fdividef(1.f, s3);
      for (int i = 0; i < stride; ++i) ra_s[i] = i < n ? ra_s[i] * inv3 : 0.f;
      if (choice) choice[q0 + lane] = arg;
    }
  }
  }
  __syncwarp();

  // write back: the tile's rows are one contiguous span of nv * stride floats
  float *pc = p_cal + q0 * stride;
  float *pa = p_avg ? p_avg + q0 * stride : nullptr;
  const int span = nv * stride;
#pragma unroll
  for (int j = 0; j < K; ++j) {
    const int e = lane + 32 * j;
    if (j < stride && e < span) {
      const int qq = (int)(((uint32_t)e * magic) >> 16);
      const int i = e - qq * stride;
      pc[e] = sa[qq * pitch + i];
      if (pa) pa[e] = sb[qq * pitch + i];
    }
  }
}

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
    const size_t smem = (size_t)kTileWarps * 64 * pitch * sizeof(float);
    // launched to overlap the previous kernel's tail; the kernels wait for it before reading
    const bool loops = n_q >= kLoopQuestions;
    auto kern = stride <= 16 ? (loops ? readout_tile_kernel<16, true> : readout_tile_kernel<16, false>)
                             : (loops ? readout_tile_kernel<32, true> : readout_tile_kernel<32, false>);
    const cudaError_t e = launch_dependent(kern, dim3(blocks), dim3(kTileWarps * 32), smem, s, logits, stride, pitch,
                                           magic, r1, r2, n_letters, temperature, n_q, p_cal, p_avg, choice, status);
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
