// tree_runtime: the whole hot path of one batch in one call, for callers that
// run batch after batch on one stream.
//
//   plan (host) -> plan image to the device -> per chunk: RoPE, attention ->
//   readout/calibration
//
// Each step packs the batch with the host planner, copies the plan image into
// one of two page-locked staging buffers, and enqueues on the caller's stream:
// a small kernel that copies the image from the staging buffer (read over the
// host link) into one of two device image buffers, then tree_rope and
// tree_attn_fwd for every chunk, then readout_decide.  Everything is one chain
// of kernels on one stream, each launched to overlap its predecessor's tail and
// waiting for it (griddepcontrol) before reading its results; there is no copy
// engine and no second stream in the step.  The two buffers alternate between
// steps: a staging buffer is rewritten only after the copy kernel that read it
// two steps earlier has run (an event, normally long passed), and a device
// image is rewritten only by a kernel that waits for the previous step's last
// kernel, so the host can plan the next batch while the GPU runs this one.
//
// Host-buffer steps (tree_runtime_step_host) add two device sets of inputs and
// outputs, used in turn, and a copy stream: the inputs of a step go host ->
// set b on the copy stream once the step two calls back has finished with set
// b, the step itself waits for them, and its decisions come back on the
// caller's stream.  So a caller that issues batch s+1 before waiting for batch
// s has the upload of s+1 running under the compute of s.

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "sm103.cuh"

struct tree_runtime {
  size_t cap = 0;  // bytes per plan image
  int32_t max_chunks = 0;
  void *dev_image[2] = {nullptr, nullptr};
  void *staging[2] = {nullptr, nullptr};     // page-locked host memory
  void *staging_dev[2] = {nullptr, nullptr}; // the same memory as the device sees it
  cudaEvent_t fetched[2] = {nullptr, nullptr};
  int32_t *work = nullptr;                   // device int32[2 * max_chunks]: attention work counters
  uint64_t steps = 0;
  // host-buffer steps
  struct IoSet {
    void *q = nullptr, *k = nullptr, *v = nullptr, *o = nullptr;
    float *logits = nullptr, *temp = nullptr, *p_cal = nullptr, *p_avg = nullptr;
    int32_t *n = nullptr, *choice = nullptr;
  };
  bool has_io = false;
  tree_io_caps_t caps = {};
  IoSet io[2];
  cudaStream_t copy = nullptr;
  cudaEvent_t uploaded[2] = {nullptr, nullptr};  // the copies into set b have run (copy stream)
  cudaEvent_t consumed[2] = {nullptr, nullptr};  // the step that used set b, and its copies back, have run
  uint64_t io_steps = 0;
};

namespace tree {
namespace {

// Copies the plan image from page-locked staging into a device buffer.  It does
// not wait for the kernel before it (the previous step's readout): it starts
// only once that readout has passed its own wait for the previous step's
// attention, and the buffer it writes was last read by the step before, which
// had completed before the previous step's RoPE passed its wait.  So the copy,
// and then this step's RoPE (which waits for the copy), overlap the readout.
__global__ void __launch_bounds__(256) fetch_image(const int4 *__restrict__ src, int4 *__restrict__ dst, int n16) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += gridDim.x * blockDim.x) dst[i] = src[i];
}

void release_io(tree_runtime *rt) {
  for (int b = 0; b < 2; ++b) {
    tree_runtime::IoSet &x = rt->io[b];
    for (void *p : {x.q, x.k, x.v, x.o, (void *)x.logits, (void *)x.temp, (void *)x.p_cal, (void *)x.p_avg,
                    (void *)x.n, (void *)x.choice})
      if (p) cudaFree(p);
    x = tree_runtime::IoSet{};
    if (rt->uploaded[b]) cudaEventDestroy(rt->uploaded[b]);
    if (rt->consumed[b]) cudaEventDestroy(rt->consumed[b]);
    rt->uploaded[b] = rt->consumed[b] = nullptr;
  }
  if (rt->copy) cudaStreamDestroy(rt->copy);
  rt->copy = nullptr;
  rt->has_io = false;
}

void release(tree_runtime *rt) {
  release_io(rt);
  for (int k = 0; k < 2; ++k) {
    if (rt->dev_image[k]) cudaFree(rt->dev_image[k]);
    if (rt->staging[k]) cudaFreeHost(rt->staging[k]);
    if (rt->fetched[k]) cudaEventDestroy(rt->fetched[k]);
  }
  if (rt->work) cudaFree(rt->work);
  delete rt;
}

// Everything of a step after planning: the plan image to the device, RoPE and
// attention per chunk, readout.  `a` holds device buffers.
int enqueue_step(tree_runtime *rt, tree_plan_t *plan, const tree_step_args_t *a, tree_stream_t stream) {
  const Plan &P = plan->p;
  const size_t bytes = P.image.size() * sizeof(int32_t);
  if (bytes > rt->cap)
    return fail(TREE_ERR_UNSUPPORTED, "tree_runtime_step: plan image of %zu bytes > capacity %zu", bytes, rt->cap);
  if (P.n_chunks > rt->max_chunks)
    return fail(TREE_ERR_UNSUPPORTED, "tree_runtime_step: %d chunks > capacity %d", P.n_chunks, rt->max_chunks);
  if (P.n_questions > 0 && (!a->logits || !a->n_letters || !a->temperature || !a->p_cal))
    return fail(TREE_ERR_INVALID_ARG, "tree_runtime_step: the batch has questions but no readout buffers");
  const cudaStream_t s = as_stream(stream);
  const int k = (int)(rt->steps & 1);
  // the copy kernel that read staging[k] two steps ago has run
  cudaError_t e = cudaEventSynchronize(rt->fetched[k]);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_runtime_step: %s", cudaGetErrorString(e));
  std::memcpy(rt->staging[k], P.image.data(), bytes);
  const int n16 = (int)(bytes / 16);
  e = launch_dependent(fetch_image, dim3((unsigned)std::min(152, (n16 + 255) / 256)), dim3(256), 0, s,
                       reinterpret_cast<const int4 *>(rt->staging_dev[k]), reinterpret_cast<int4 *>(rt->dev_image[k]),
                       n16);
  if (e == cudaSuccess) e = cudaEventRecord(rt->fetched[k], s);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_runtime_step: %s", cudaGetErrorString(e));
  ++rt->steps;
  const void *img = rt->dev_image[k];
  const size_t qrow = (size_t)a->hq * a->d * 2;  // bytes per query row
  int rc;
  for (int c = 0; c < P.n_chunks; ++c) {
    const int32_t q0 = P.chunk_q0[c];
    void *qc = static_cast<uint8_t *>(a->q) + (size_t)(q0 - P.n_res) * qrow;
    void *oc = static_cast<uint8_t *>(a->o) + (size_t)(q0 - P.n_res) * qrow;
    float *lc = a->lse ? a->lse + (size_t)(q0 - P.n_res) * a->hq : nullptr;
    rc = tree_rope(plan, img, c, qc, a->k, a->hq, a->hkv, a->d, a->cos_sin, a->max_pos, a->status, stream);
    if (rc != TREE_OK) return rc;
    tree_attn_params_t ap = {a->hq, a->hkv, a->d, a->scale, rt->work + 2 * c, 0};
    if (c == 0 && a->attn_events[0] &&
        (e = cudaEventRecord(static_cast<cudaEvent_t>(a->attn_events[0]), s)) != cudaSuccess)
      return fail(TREE_ERR_CUDA, "tree_runtime_step: %s", cudaGetErrorString(e));
    rc = tree_attn_fwd(plan, img, c, qc, a->k, a->v, oc, lc, &ap, a->status, stream);
    if (rc != TREE_OK) return rc;
    if (c == P.n_chunks - 1 && a->attn_events[1] &&
        (e = cudaEventRecord(static_cast<cudaEvent_t>(a->attn_events[1]), s)) != cudaSuccess)
      return fail(TREE_ERR_CUDA, "tree_runtime_step: %s", cudaGetErrorString(e));
  }
  if (P.n_questions > 0) {
    const int32_t *base = static_cast<const int32_t *>(img);
    rc = readout_decide(a->logits, a->stride, base + P.off_r1, base + P.off_r2, a->n_letters, a->temperature,
                        P.n_questions, a->p_cal, a->p_avg, a->choice, a->status, stream);
    if (rc != TREE_OK) return rc;
  }
  return TREE_OK;
}

struct PlanGuard {
  tree_plan_t *p = nullptr;
  ~PlanGuard() { tree_plan_free(p); }
};

}  // namespace
}  // namespace tree

extern "C" TREE_API int tree_runtime_create(size_t max_plan_bytes, int32_t max_chunks, tree_runtime_t **out) {
  using namespace tree;
  if (!out || max_plan_bytes == 0 || max_chunks <= 0)
    return fail(TREE_ERR_INVALID_ARG, "tree_runtime_create: max_plan_bytes %zu, max_chunks %d", max_plan_bytes,
                max_chunks);
  *out = nullptr;
  auto *rt = new tree_runtime;
  rt->cap = (max_plan_bytes + 15) / 16 * 16;
  rt->max_chunks = max_chunks;
  cudaError_t e = cudaSuccess;
  for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
    e = cudaMalloc(&rt->dev_image[k], rt->cap);
    if (e == cudaSuccess) e = cudaHostAlloc(&rt->staging[k], rt->cap, cudaHostAllocMapped);
    if (e == cudaSuccess) e = cudaHostGetDevicePointer(&rt->staging_dev[k], rt->staging[k], 0);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&rt->fetched[k], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaMalloc(&rt->work, sizeof(int32_t) * 2 * (size_t)max_chunks);
  if (e == cudaSuccess) e = cudaMemset(rt->work, 0, sizeof(int32_t) * 2 * (size_t)max_chunks);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();  // the counters are zero before any step
  if (e != cudaSuccess) {
    release(rt);
    return fail(TREE_ERR_CUDA, "tree_runtime_create: %s", cudaGetErrorString(e));
  }
  *out = rt;
  return TREE_OK;
}

extern "C" TREE_API int tree_runtime_destroy(tree_runtime_t *rt) {
  if (!rt) return TREE_OK;
  // buffers may still be in use by queued work
  for (int k = 0; k < 2; ++k)
    if (rt->fetched[k]) cudaEventSynchronize(rt->fetched[k]);
  cudaDeviceSynchronize();
  tree::release(rt);
  return TREE_OK;
}

extern "C" TREE_API int tree_runtime_step(tree_runtime_t *rt, const tree_step_args_t *a, tree_plan_info_t *info_out,
                                          tree_stream_t stream) {
  using namespace tree;
  if (!rt || !a || !a->spec || !a->q || !a->k || !a->v || !a->o || !a->cos_sin)
    return fail(TREE_ERR_INVALID_ARG, "tree_runtime_step: NULL argument");
  PlanGuard guard;
  int rc = tree_pack_plan(a->spec, a->opts, &guard.p);
  if (rc != TREE_OK) return rc;
  rc = enqueue_step(rt, guard.p, a, stream);
  if (rc != TREE_OK) return rc;
  if (info_out) return tree_plan_query(guard.p, info_out);
  return TREE_OK;
}

extern "C" TREE_API int tree_runtime_attach_io(tree_runtime_t *rt, const tree_io_caps_t *caps) {
  using namespace tree;
  if (!rt || !caps) return fail(TREE_ERR_INVALID_ARG, "tree_runtime_attach_io: NULL argument");
  const tree_io_caps_t &c = *caps;
  if (c.max_fwd <= 0 || c.max_tot < c.max_fwd || c.hq <= 0 || c.hkv <= 0 || c.hq % c.hkv != 0 || c.d <= 0 ||
      c.stride < 0 || c.max_slots < 0 || c.max_questions < 0 ||
      (c.stride == 0 && (c.max_slots > 0 || c.max_questions > 0)))
    return fail(TREE_ERR_INVALID_ARG,
                "tree_runtime_attach_io: max_fwd %d, max_tot %d, hq %d, hkv %d, d %d, stride %d, max_slots %d, "
                "max_questions %d",
                c.max_fwd, c.max_tot, c.hq, c.hkv, c.d, c.stride, c.max_slots, c.max_questions);
  // the old sets may still be in use by queued work
  cudaError_t e = cudaDeviceSynchronize();
  release_io(rt);
  const size_t qb = (size_t)c.max_fwd * c.hq * c.d * 2, kb = (size_t)c.max_tot * c.hkv * c.d * 2;
  const size_t lb = (size_t)c.max_slots * c.stride * 4, nb = (size_t)c.max_questions * 4;
  const size_t pb = (size_t)c.max_questions * c.stride * 4;
  for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
    tree_runtime::IoSet &x = rt->io[b];
    e = cudaMalloc(&x.q, qb);
    if (e == cudaSuccess) e = cudaMalloc(&x.k, kb);
    if (e == cudaSuccess) e = cudaMalloc(&x.v, kb);
    if (e == cudaSuccess) e = cudaMalloc(&x.o, qb);
    if (e == cudaSuccess && lb) e = cudaMalloc(&x.logits, lb);
    if (e == cudaSuccess && nb) e = cudaMalloc(&x.temp, nb);
    if (e == cudaSuccess && nb) e = cudaMalloc(&x.n, nb);
    if (e == cudaSuccess && nb) e = cudaMalloc(&x.choice, nb);
    if (e == cudaSuccess && pb) e = cudaMalloc(&x.p_cal, pb);
    if (e == cudaSuccess && pb) e = cudaMalloc(&x.p_avg, pb);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&rt->uploaded[b], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&rt->consumed[b], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&rt->copy, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    release_io(rt);
    return fail(TREE_ERR_CUDA, "tree_runtime_attach_io: %s", cudaGetErrorString(e));
  }
  rt->caps = c;
  rt->has_io = true;
  rt->io_steps = 0;
  return TREE_OK;
}

extern "C" TREE_API int tree_runtime_step_host(tree_runtime_t *rt, const tree_host_step_args_t *a,
                                               tree_plan_info_t *info_out, tree_stream_t stream) {
  using namespace tree;
  if (!rt || !a || !a->spec || !a->q || !a->k || !a->v || !a->cos_sin)
    return fail(TREE_ERR_INVALID_ARG, "tree_runtime_step_host: NULL argument");
  if (!rt->has_io) return fail(TREE_ERR_INVALID_ARG, "tree_runtime_step_host: no buffers attached");
  PlanGuard guard;
  int rc = tree_pack_plan(a->spec, a->opts, &guard.p);
  if (rc != TREE_OK) return rc;
  const Plan &P = guard.p->p;
  const tree_io_caps_t &c = rt->caps;
  const int32_t n_fwd = P.n_tot - P.n_res, n_slots = (int32_t)P.slot_tok.size();
  if (n_fwd > c.max_fwd || P.n_tot > c.max_tot)
    return fail(TREE_ERR_INVALID_ARG, "tree_runtime_step_host: %d forward / %d key rows > capacity %d / %d", n_fwd,
                P.n_tot, c.max_fwd, c.max_tot);
  const int32_t nq = P.n_questions;
  if (nq > 0) {
    if (!a->logits || !a->n_letters || !a->temperature)
      return fail(TREE_ERR_INVALID_ARG, "tree_runtime_step_host: the batch has questions but no readout inputs");
    if (n_slots > c.max_slots || nq > c.max_questions)
      return fail(TREE_ERR_INVALID_ARG, "tree_runtime_step_host: %d slots / %d questions > capacity %d / %d",
                  n_slots, nq, c.max_slots, c.max_questions);
  }
  const cudaStream_t s = as_stream(stream);
  const int b = (int)(rt->io_steps & 1);
  tree_runtime::IoSet &x = rt->io[b];
  const size_t qb = (size_t)n_fwd * c.hq * c.d * 2, kb = (size_t)P.n_tot * c.hkv * c.d * 2;
  const size_t pb = (size_t)nq * c.stride * 4;
  // upload on the copy stream, once the step two calls back is done with set b
  cudaError_t e = cudaStreamWaitEvent(rt->copy, rt->consumed[b], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(x.q, a->q, qb, cudaMemcpyHostToDevice, rt->copy);
  if (e == cudaSuccess) e = cudaMemcpyAsync(x.k, a->k, kb, cudaMemcpyHostToDevice, rt->copy);
  if (e == cudaSuccess) e = cudaMemcpyAsync(x.v, a->v, kb, cudaMemcpyHostToDevice, rt->copy);
  if (e == cudaSuccess && nq > 0)
    e = cudaMemcpyAsync(x.logits, a->logits, (size_t)n_slots * c.stride * 4, cudaMemcpyHostToDevice, rt->copy);
  if (e == cudaSuccess && nq > 0) e = cudaMemcpyAsync(x.n, a->n_letters, (size_t)nq * 4, cudaMemcpyHostToDevice, rt->copy);
  if (e == cudaSuccess && nq > 0)
    e = cudaMemcpyAsync(x.temp, a->temperature, (size_t)nq * 4, cudaMemcpyHostToDevice, rt->copy);
  if (e == cudaSuccess) e = cudaEventRecord(rt->uploaded[b], rt->copy);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, rt->uploaded[b], 0);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_runtime_step_host: %s", cudaGetErrorString(e));
  ++rt->io_steps;

  tree_step_args_t d = {};
  d.spec = a->spec;
  d.opts = a->opts;
  d.q = x.q;
  d.k = x.k;
  d.v = x.v;
  d.o = x.o;
  d.cos_sin = a->cos_sin;
  d.max_pos = a->max_pos;
  d.hq = c.hq;
  d.hkv = c.hkv;
  d.d = c.d;
  d.scale = a->scale;
  if (nq > 0) {
    d.logits = x.logits;
    d.stride = c.stride;
    d.n_letters = x.n;
    d.temperature = x.temp;
    d.p_cal = x.p_cal;
    d.p_avg = a->p_avg ? x.p_avg : nullptr;
    d.choice = x.choice;
  }
  d.status = a->status;
  rc = enqueue_step(rt, guard.p, &d, stream);
  if (rc != TREE_OK) return rc;
  // results back on the caller's stream (each copy waits for the step's last kernel)
  if (nq > 0 && a->choice) e = cudaMemcpyAsync(a->choice, x.choice, (size_t)nq * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && nq > 0 && a->p_cal) e = cudaMemcpyAsync(a->p_cal, x.p_cal, pb, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && nq > 0 && a->p_avg) e = cudaMemcpyAsync(a->p_avg, x.p_avg, pb, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && a->o) e = cudaMemcpyAsync(a->o, x.o, qb, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaEventRecord(rt->consumed[b], s);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_runtime_step_host: %s", cudaGetErrorString(e));
  if (info_out) return tree_plan_query(guard.p, info_out);
  return TREE_OK;
}
