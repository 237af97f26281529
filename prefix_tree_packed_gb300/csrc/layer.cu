// tree_layer_fwd: one Llama layer over the packed forward tokens of a batch,
// as a chain of the library's kernels on one stream (basal-rs Architecture
// page, "01 / Request path: GPU forward pass": the Llama model in f16 over the
// batch as one compact token list; attention over tree blocks per "03 /
// Packing").  The projections run over all forward tokens at once; RoPE and
// attention run per forward chunk (chunk c reads the keys of chunks <= c,
// which earlier iterations have rotated).

#include <chrono>
#include <vector>

#include "common.cuh"
#include "sm103.cuh"
#include "tree_layer.h"

namespace tree {
namespace {

struct LayerWs {
  size_t xn, q, o, h, g, total;  // byte offsets of the f16 buffers
};

inline size_t up256(size_t b) { return (b + 255) & ~size_t(255); }

LayerWs layout(int64_t n_fwd, const tree_layer_weights_t &w) {
  LayerWs L;
  const size_t e = 2;
  L.xn = 0;
  L.q = L.xn + up256((size_t)n_fwd * w.hidden * e);
  L.o = L.q + up256((size_t)n_fwd * w.hq * w.d * e);
  L.h = L.o + up256((size_t)n_fwd * w.hq * w.d * e);
  L.g = L.h + up256((size_t)n_fwd * w.hidden * e);
  L.total = L.g + up256((size_t)n_fwd * w.ffn * e);
  return L;
}

// Last layer: the attention block over every token (the keys and values of all
// of them are needed), then only the readout rows (one per readout slot).
struct LastWs {
  size_t xn, q, o, xs, os, hs, hns, gs, ys, fs, total;
};

LastWs last_layout(int64_t n_fwd, int64_t n_slots, const tree_layer_weights_t &w) {
  LastWs L;
  const size_t e = 2, S = (size_t)n_slots;
  L.xn = 0;
  L.q = L.xn + up256((size_t)n_fwd * w.hidden * e);
  L.o = L.q + up256((size_t)n_fwd * w.hq * w.d * e);
  L.xs = L.o + up256((size_t)n_fwd * w.hq * w.d * e);
  L.os = L.xs + up256(S * w.hidden * e);
  L.hs = L.os + up256(S * w.hq * w.d * e);
  L.hns = L.hs + up256(S * w.hidden * e);
  L.gs = L.hns + up256(S * w.hidden * e);
  L.ys = L.gs + up256(S * w.ffn * e);
  L.fs = L.ys + up256(S * w.hidden * e);
  L.total = L.fs + up256(S * w.hidden * e);
  return L;
}

constexpr int kGatherWarps = 8;

// dst[i, :] = src[slot_tok[i] - n_res, :] for the readout slots (rows of 16-byte vectors)
__global__ void __launch_bounds__(kGatherWarps * 32) gather_slots(const uint4 *src, int vec_per_row,
                                                                   const int32_t *slot_tok, int n_res, uint4 *dst,
                                                                   int m) {
  sm103::griddep_wait();
  sm103::griddep_launch();
  const int row = blockIdx.x * kGatherWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= m) return;
  const size_t s = (size_t)(slot_tok[row] - n_res);
  // chunks of 8 loads per lane in flight before their stores (dst never overlaps src)
  for (int i0 = 0; i0 < vec_per_row; i0 += 256) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + lane + 32 * u;
      if (i < vec_per_row) v[u] = src[s * vec_per_row + i];
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + lane + 32 * u;
      if (i < vec_per_row) dst[(size_t)row * vec_per_row + i] = v[u];
    }
  }
}

int gather(const __half *src, int cols, const int32_t *slot_tok, int n_res, __half *dst, int m, cudaStream_t s) {
  if (m == 0) return TREE_OK;
  const cudaError_t e = launch_dependent(gather_slots, dim3((m + kGatherWarps - 1) / kGatherWarps),
                                         dim3(kGatherWarps * 32), 0, s, reinterpret_cast<const uint4 *>(src),
                                         cols / 8, slot_tok, n_res, reinterpret_cast<uint4 *>(dst), m);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "tree_last_layer_fwd: launch failed: %s", cudaGetErrorString(e));
  return launch_status("tree_last_layer_fwd");
}

int check_weights(const tree_layer_weights_t *w) {
  if (!w) return fail(TREE_ERR_INVALID_ARG, "tree_layer: NULL weights");
  if (w->hidden <= 0 || w->hq <= 0 || w->hkv <= 0 || w->ffn <= 0 || w->hq % w->hkv)
    return fail(TREE_ERR_INVALID_ARG, "tree_layer: hidden %d, hq %d, hkv %d, ffn %d", w->hidden, w->hq, w->hkv, w->ffn);
  if (w->d != 64 && w->d != 128) return fail(TREE_ERR_UNSUPPORTED, "tree_layer: head dim %d", w->d);
  if (w->hidden % 8 || w->ffn % 8) return fail(TREE_ERR_UNSUPPORTED, "tree_layer: hidden and ffn must be multiples of 8");
  if (!w->w_in || !w->wqkv || !w->wo || !w->w_post || !w->wgu || !w->wd)
    return fail(TREE_ERR_INVALID_ARG, "tree_layer: NULL weight");
  return TREE_OK;
}

}  // namespace
}  // namespace tree

extern "C" TREE_API int tree_layer_workspace_bytes(const tree_plan_t *plan, const tree_layer_weights_t *w,
                                                   size_t *bytes) {
  using namespace tree;
  if (!plan || !bytes) return fail(TREE_ERR_INVALID_ARG, "tree_layer_workspace_bytes: NULL argument");
  int rc = check_weights(w);
  if (rc) return rc;
  *bytes = layout(plan->p.n_tot - plan->p.n_res, *w).total;
  return TREE_OK;
}

extern "C" TREE_API int tree_layer_fwd(const tree_plan_t *plan, const void *plan_dev, const tree_layer_weights_t *w,
                                       const void *x, void *k_cache, void *v_cache, void *y, const float *cos_sin,
                                       int32_t max_pos, void *workspace, size_t workspace_bytes, int32_t *work,
                                       int32_t *status, tree_stream_t stream) {
  using namespace tree;
  if (!plan || !plan_dev || !x || !k_cache || !v_cache || !y || !cos_sin || !workspace)
    return fail(TREE_ERR_INVALID_ARG, "tree_layer_fwd: NULL argument");
  int rc = check_weights(w);
  if (rc) return rc;
  if (x == y) return fail(TREE_ERR_INVALID_ARG, "tree_layer_fwd: y may not alias x");
  const Plan &P = plan->p;
  const int64_t n_fwd = P.n_tot - P.n_res;
  const LayerWs L = layout(n_fwd, *w);
  if (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return fail(TREE_ERR_INVALID_ARG, "tree_layer_fwd: workspace of %zu bytes (need %zu, 256-byte aligned)",
                workspace_bytes, L.total);
  if (n_fwd == 0) return TREE_OK;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  __half *xn = reinterpret_cast<__half *>(ws + L.xn), *q = reinterpret_cast<__half *>(ws + L.q);
  __half *o = reinterpret_cast<__half *>(ws + L.o), *h = reinterpret_cast<__half *>(ws + L.h);
  __half *g = reinterpret_cast<__half *>(ws + L.g);
  const int qd = w->hq * w->d, kvd = w->hkv * w->d, m = (int)n_fwd;
  __half *kf = static_cast<__half *>(k_cache) + (size_t)P.n_res * kvd;
  __half *vf = static_cast<__half *>(v_cache) + (size_t)P.n_res * kvd;
  // attention block
  if ((rc = tree_rmsnorm(x, w->w_in, xn, m, w->hidden, w->eps, stream))) return rc;
  if ((rc = tree_gemm_qkv(xn, w->wqkv, q, kf, vf, m, qd, kvd, w->hidden, status, stream))) return rc;
  tree_attn_params_t ap{w->hq, w->hkv, w->d, 0.f, nullptr, 0};
  for (int c = 0; c < P.n_chunks; ++c) {
    const size_t r0 = (size_t)(P.chunk_q0[c] - P.n_res);
    if ((rc = tree_rope(plan, plan_dev, c, q + r0 * qd, k_cache, w->hq, w->hkv, w->d, cos_sin, max_pos, status,
                        stream)))
      return rc;
    ap.work = work ? work + 2 * c : nullptr;
    if ((rc = tree_attn_fwd(plan, plan_dev, c, q + r0 * qd, k_cache, v_cache, o + r0 * qd, nullptr, &ap, status,
                            stream)))
      return rc;
  }
  if ((rc = tree_gemm(o, w->wo, h, x, m, w->hidden, qd, TREE_GEMM_RESIDUAL, status, stream))) return rc;
  // MLP block
  if ((rc = tree_rmsnorm(h, w->w_post, xn, m, w->hidden, w->eps, stream))) return rc;
  if ((rc = tree_gemm(xn, w->wgu, g, nullptr, m, w->ffn, w->hidden, TREE_GEMM_SWIGLU, status, stream))) return rc;
  return tree_gemm(g, w->wd, y, h, m, w->hidden, w->ffn, TREE_GEMM_RESIDUAL, status, stream);
}

extern "C" TREE_API int tree_last_layer_workspace_bytes(const tree_plan_t *plan, const tree_layer_weights_t *w,
                                                        size_t *bytes) {
  using namespace tree;
  if (!plan || !bytes) return fail(TREE_ERR_INVALID_ARG, "tree_last_layer_workspace_bytes: NULL argument");
  int rc = check_weights(w);
  if (rc) return rc;
  *bytes = last_layout(plan->p.n_tot - plan->p.n_res, (int64_t)plan->p.slot_tok.size(), *w).total;
  return TREE_OK;
}

extern "C" TREE_API int tree_last_layer_fwd(const tree_plan_t *plan, const void *plan_dev,
                                            const tree_layer_weights_t *w, const void *x, void *k_cache,
                                            void *v_cache, const float *cos_sin, int32_t max_pos, const void *w_final,
                                            const void *w_letters, int32_t stride, float *logits, void *workspace,
                                            size_t workspace_bytes, int32_t *work, int32_t *status,
                                            tree_stream_t stream) {
  using namespace tree;
  if (!plan || !plan_dev || !x || !k_cache || !v_cache || !cos_sin || !w_final || !w_letters || !logits || !workspace)
    return fail(TREE_ERR_INVALID_ARG, "tree_last_layer_fwd: NULL argument");
  int rc = check_weights(w);
  if (rc) return rc;
  if (stride <= 0 || stride % 8) return fail(TREE_ERR_UNSUPPORTED, "tree_last_layer_fwd: stride %d (multiple of 8)", stride);
  if (!aligned16(w_final) || !aligned16(w_letters) || !aligned16(logits))
    return fail(TREE_ERR_UNSUPPORTED, "tree_last_layer_fwd: misaligned pointer");
  const Plan &P = plan->p;
  const int64_t n_fwd = P.n_tot - P.n_res;
  const int S = (int)P.slot_tok.size();
  for (int i = 0; i < S; ++i)
    if (P.slot_tok[i] < P.n_res)
      return fail(TREE_ERR_INVALID_ARG, "tree_last_layer_fwd: readout slot %d is a resident token", i);
  const LastWs L = last_layout(n_fwd, S, *w);
  if (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return fail(TREE_ERR_INVALID_ARG, "tree_last_layer_fwd: workspace of %zu bytes (need %zu, 256-byte aligned)",
                workspace_bytes, L.total);
  if (n_fwd == 0 || S == 0) return TREE_OK;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  auto at = [&](size_t off) { return reinterpret_cast<__half *>(ws + off); };
  __half *xn = at(L.xn), *q = at(L.q), *o = at(L.o);
  __half *xs = at(L.xs), *os = at(L.os), *hs = at(L.hs), *hns = at(L.hns), *gs = at(L.gs), *ys = at(L.ys),
         *fs = at(L.fs);
  const int qd = w->hq * w->d, kvd = w->hkv * w->d, m = (int)n_fwd;
  __half *kf = static_cast<__half *>(k_cache) + (size_t)P.n_res * kvd;
  __half *vf = static_cast<__half *>(v_cache) + (size_t)P.n_res * kvd;
  const int32_t *slot_tok = reinterpret_cast<const int32_t *>(plan_dev) + P.off_slot_tok;
  const cudaStream_t s = as_stream(stream);
  // attention block over every forward token
  if ((rc = tree_rmsnorm(x, w->w_in, xn, m, w->hidden, w->eps, stream))) return rc;
  if ((rc = tree_gemm_qkv(xn, w->wqkv, q, kf, vf, m, qd, kvd, w->hidden, status, stream))) return rc;
  tree_attn_params_t ap{w->hq, w->hkv, w->d, 0.f, nullptr, 0};
  for (int c = 0; c < P.n_chunks; ++c) {
    const size_t r0 = (size_t)(P.chunk_q0[c] - P.n_res);
    if ((rc = tree_rope(plan, plan_dev, c, q + r0 * qd, k_cache, w->hq, w->hkv, w->d, cos_sin, max_pos, status,
                        stream)))
      return rc;
    ap.work = work ? work + 2 * c : nullptr;
    if ((rc = tree_attn_fwd(plan, plan_dev, c, q + r0 * qd, k_cache, v_cache, o + r0 * qd, nullptr, &ap, status,
                            stream)))
      return rc;
  }
  // from here on only the readout rows ("01 / Request path: GPU forward pass": in the final
  // layer the MLP block and the logits are computed only for readout positions and letters)
  if ((rc = gather(o, qd, slot_tok, P.n_res, os, S, s))) return rc;
  if ((rc = gather(static_cast<const __half *>(x), w->hidden, slot_tok, P.n_res, xs, S, s))) return rc;
  if ((rc = tree_gemm(os, w->wo, hs, xs, S, w->hidden, qd, TREE_GEMM_RESIDUAL, status, stream))) return rc;
  if ((rc = tree_rmsnorm(hs, w->w_post, hns, S, w->hidden, w->eps, stream))) return rc;
  if ((rc = tree_gemm(hns, w->wgu, gs, nullptr, S, w->ffn, w->hidden, TREE_GEMM_SWIGLU, status, stream))) return rc;
  if ((rc = tree_gemm(gs, w->wd, ys, hs, S, w->hidden, w->ffn, TREE_GEMM_RESIDUAL, status, stream))) return rc;
  if ((rc = tree_rmsnorm(ys, w_final, fs, S, w->hidden, w->eps, stream))) return rc;
  return tree_gemm(fs, w_letters, logits, nullptr, S, stride, w->hidden, TREE_GEMM_STORE_F32, status, stream);
}

// ---------------------------------------------------------------------------
// tree_model_fwd: layers 0 .. n-2 through tree_layer_fwd (hidden states in two
// buffers taken in turn), the last through tree_last_layer_fwd.

namespace tree {
namespace {

size_t model_bytes(const Plan &P, const tree_layer_weights_t &w) {
  const int64_t n_fwd = P.n_tot - P.n_res;
  const size_t hid = up256((size_t)n_fwd * w.hidden * 2);
  const size_t a = layout(n_fwd, w).total, b = last_layout(n_fwd, (int64_t)P.slot_tok.size(), w).total;
  return 2 * hid + (a > b ? a : b);
}

}  // namespace
}  // namespace tree

extern "C" TREE_API int tree_model_workspace_bytes(const tree_plan_t *plan, const tree_layer_weights_t *w,
                                                   size_t *bytes) {
  using namespace tree;
  if (!plan || !bytes) return fail(TREE_ERR_INVALID_ARG, "tree_model_workspace_bytes: NULL argument");
  int rc = check_weights(w);
  if (rc) return rc;
  *bytes = model_bytes(plan->p, *w);
  return TREE_OK;
}

extern "C" TREE_API int tree_model_fwd(const tree_plan_t *plan, const void *plan_dev,
                                       const tree_layer_weights_t *layers, int32_t n_layers, const void *x,
                                       void *const *k_caches, void *const *v_caches, const float *cos_sin,
                                       int32_t max_pos, const void *w_final, const void *w_letters, int32_t stride,
                                       float *logits, void *workspace, size_t workspace_bytes, int32_t *work,
                                       int32_t *status, tree_stream_t stream) {
  using namespace tree;
  if (!plan || !layers || n_layers < 1 || !x || !k_caches || !v_caches || !workspace)
    return fail(TREE_ERR_INVALID_ARG, "tree_model_fwd: NULL argument or n_layers %d", n_layers);
  const tree_layer_weights_t &w0 = layers[0];
  int rc = check_weights(&w0);
  if (rc) return rc;
  for (int l = 1; l < n_layers; ++l)
    if (layers[l].hidden != w0.hidden || layers[l].hq != w0.hq || layers[l].hkv != w0.hkv || layers[l].d != w0.d ||
        layers[l].ffn != w0.ffn)
      return fail(TREE_ERR_INVALID_ARG, "tree_model_fwd: layer %d has other sizes than layer 0", l);
  const Plan &P = plan->p;
  const size_t need = model_bytes(P, w0);
  if (workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return fail(TREE_ERR_INVALID_ARG, "tree_model_fwd: workspace of %zu bytes (need %zu, 256-byte aligned)",
                workspace_bytes, need);
  const int64_t n_fwd = P.n_tot - P.n_res;
  const size_t hid = up256((size_t)n_fwd * w0.hidden * 2);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  void *buf[2] = {ws, ws + hid};
  uint8_t *inner = ws + 2 * hid;
  const size_t inner_bytes = workspace_bytes - 2 * hid;
  const void *cur = x;
  for (int l = 0; l + 1 < n_layers; ++l) {
    void *next = buf[l & 1];
    if ((rc = tree_layer_fwd(plan, plan_dev, &layers[l], cur, k_caches[l], v_caches[l], next, cos_sin, max_pos,
                             inner, inner_bytes, work, status, stream)))
      return rc;
    cur = next;
  }
  const int l = n_layers - 1;
  return tree_last_layer_fwd(plan, plan_dev, &layers[l], cur, k_caches[l], v_caches[l], cos_sin, max_pos, w_final,
                             w_letters, stride, logits, inner, inner_bytes, work, status, stream);
}

// ---------------------------------------------------------------------------
// Long-lane sessions: tree_model_fwd's layer loop, resumable between layers.

struct tree_session {
  const tree_plan_t *plan = nullptr;
  const void *plan_dev = nullptr;
  std::vector<tree_layer_weights_t> layers;
  std::vector<void *> kc, vc;
  const void *x = nullptr;
  const float *cos_sin = nullptr;
  int32_t max_pos = 0, stride = 0;
  const void *w_final = nullptr, *w_letters = nullptr;
  float *logits = nullptr;
  uint8_t *ws = nullptr;
  size_t ws_bytes = 0, hid = 0;
  int32_t *work = nullptr, *status = nullptr;
  int next = 0;  // the next layer to run
  cudaEvent_t ev = nullptr;
};

extern "C" TREE_API int tree_session_create(const tree_plan_t *plan, const void *plan_dev,
                                            const tree_layer_weights_t *layers, int32_t n_layers, const void *x,
                                            void *const *k_caches, void *const *v_caches, const float *cos_sin,
                                            int32_t max_pos, const void *w_final, const void *w_letters,
                                            int32_t stride, float *logits, void *workspace, size_t workspace_bytes,
                                            int32_t *work, int32_t *status, tree_session_t **out) {
  using namespace tree;
  if (!out) return fail(TREE_ERR_INVALID_ARG, "tree_session_create: NULL out");
  *out = nullptr;
  if (!plan || !plan_dev || !layers || n_layers < 1 || !x || !k_caches || !v_caches || !cos_sin || !w_final ||
      !w_letters || !logits || !workspace)
    return fail(TREE_ERR_INVALID_ARG, "tree_session_create: NULL argument or n_layers %d", n_layers);
  int rc = check_weights(&layers[0]);
  if (rc) return rc;
  const size_t need = model_bytes(plan->p, layers[0]);
  if (workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return fail(TREE_ERR_INVALID_ARG, "tree_session_create: workspace of %zu bytes (need %zu, 256-byte aligned)",
                workspace_bytes, need);
  auto *s = new tree_session;
  s->plan = plan;
  s->plan_dev = plan_dev;
  s->layers.assign(layers, layers + n_layers);
  s->kc.assign(k_caches, k_caches + n_layers);
  s->vc.assign(v_caches, v_caches + n_layers);
  s->x = x;
  s->cos_sin = cos_sin;
  s->max_pos = max_pos;
  s->w_final = w_final;
  s->w_letters = w_letters;
  s->stride = stride;
  s->logits = logits;
  s->ws = static_cast<uint8_t *>(workspace);
  s->ws_bytes = workspace_bytes;
  s->hid = up256((size_t)(plan->p.n_tot - plan->p.n_res) * layers[0].hidden * 2);
  s->work = work;
  s->status = status;
  const cudaError_t e = cudaEventCreateWithFlags(&s->ev, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    delete s;
    return fail(TREE_ERR_CUDA, "tree_session_create: %s", cudaGetErrorString(e));
  }
  *out = s;
  return TREE_OK;
}

extern "C" TREE_API int tree_session_run(tree_session_t *s, double slice_ms, tree_stream_t stream,
                                         int32_t *layers_run, int32_t *done) {
  using namespace tree;
  if (!s) return fail(TREE_ERR_INVALID_ARG, "tree_session_run: NULL session");
  const int n = (int)s->layers.size();
  int ran = 0;
  const auto t0 = std::chrono::steady_clock::now();
  void *buf[2] = {s->ws, s->ws + s->hid};
  uint8_t *inner = s->ws + 2 * s->hid;
  const size_t inner_bytes = s->ws_bytes - 2 * s->hid;
  int rc = TREE_OK;
  while (s->next < n) {
    const int l = s->next;
    // layer l reads the input (l = 0) or the buffer layer l - 1 wrote, exactly as in tree_model_fwd
    const void *cur = l == 0 ? s->x : buf[(l - 1) & 1];
    if (l + 1 < n)
      rc = tree_layer_fwd(s->plan, s->plan_dev, &s->layers[l], cur, s->kc[l], s->vc[l], buf[l & 1], s->cos_sin,
                          s->max_pos, inner, inner_bytes, s->work, s->status, stream);
    else
      rc = tree_last_layer_fwd(s->plan, s->plan_dev, &s->layers[l], cur, s->kc[l], s->vc[l], s->cos_sin, s->max_pos,
                               s->w_final, s->w_letters, s->stride, s->logits, inner, inner_bytes, s->work, s->status,
                               stream);
    if (rc) break;
    ++s->next;
    ++ran;
    // the layer's end, then the slice check: yield once the slice is used up
    cudaError_t e = cudaEventRecord(s->ev, as_stream(stream));
    if (e == cudaSuccess) e = cudaEventSynchronize(s->ev);
    if (e != cudaSuccess) {
      rc = fail(TREE_ERR_CUDA, "tree_session_run: %s", cudaGetErrorString(e));
      break;
    }
    const double ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    if (ms >= slice_ms) break;
  }
  if (layers_run) *layers_run = ran;
  if (done) *done = s->next >= n ? 1 : 0;
  return rc;
}

extern "C" TREE_API int tree_session_destroy(tree_session_t *s) {
  if (s) {
    if (s->ev) cudaEventDestroy(s->ev);
    delete s;
  }
  return TREE_OK;
}
