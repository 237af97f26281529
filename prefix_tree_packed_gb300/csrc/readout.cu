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
//
// Work layout: a group of G lanes per question, each lane holding letters
// lane, lane + G, ...  G = 32 (one warp per question, up to 255 letters) in
// general; G = 1 (one lane per question, no shuffles) when every question has
// at most 16 letters, i.e. stride <= 16, which makes the kernel bound by HBM
// rather than by shuffle latency on batches of small questions.

#include <cfloat>

#include "common.cuh"

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
      x1[k] = expf(x1[k] - m1);
      x2[k] = expf(x2[k] - m2);
      s1 += x1[k];
      s2 += x2[k];
    }
  }
  s1 = group_sum<G>(s1);
  s2 = group_sum<G>(s2);
  const float inv1 = 1.f / s1, inv2 = 1.f / s2, invT = 1.f / T;
  // p (kept in x1), its calibrated logit (kept in x2), argmax of p
  float m3 = -FLT_MAX, best = -1.f;
  int arg = 0x7fffffff;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int i = lane + G * k;
    if (i < n) {
      const float p = 0.5f * (x1[k] * inv1 + x2[k] * inv2);
      x1[k] = p;
      x2[k] = logf(fmaxf(p, kClamp)) * invT;
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
      x2[k] = expf(x2[k] - m3);
      s3 += x2[k];
    }
  }
  s3 = group_sum<G>(s3);
  const float inv3 = 1.f / s3;
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
  if (stride <= 16) {
    const int threads = 256;
    const int blocks = (int)(((int64_t)n_q + threads - 1) / threads);
    readout_kernel<1, 16><<<blocks, threads, 0, s>>>(logits, stride, r1, r2, n_letters, temperature, n_q,
                                                     p_cal, p_avg, choice, status);
  } else {
    const int threads = 256;
    const int64_t lanes = (int64_t)n_q * 32;
    const int blocks = (int)((lanes + threads - 1) / threads);
    readout_kernel<32, 8><<<blocks, threads, 0, s>>>(logits, stride, r1, r2, n_letters, temperature, n_q,
                                                     p_cal, p_avg, choice, status);
  }
  return launch_status("readout_decide");
}
