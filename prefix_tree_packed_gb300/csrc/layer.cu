// tree_layer_fwd: one Llama layer over the packed forward tokens of a batch,
// as a chain of the library's kernels on one stream (basal-rs Architecture
// page, "01 / Request path: GPU forward pass": the Llama model in f16 over the
// batch as one compact token list; attention over tree blocks per "03 /
// Packing").  The projections run over all forward tokens at once; RoPE and
// attention run per forward chunk (chunk c reads the keys of chunks <= c,
// which earlier iterations have rotated).

#include "common.cuh"
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

int check_weights(const tree_layer_weights_t *w) {
  if (!w) return fail(TREE_ERR_INVALID_ARG, "tree_layer: NULL weights");
  if (w->hidden <= 0 || w->hq <= 0 || w->hkv <= 0 || w->ffn <= 0 || w->hq % w->hkv)
    return fail(TREE_ERR_INVALID_ARG, "tree_layer: hidden %d, hq %d, hkv %d, ffn %d", w->hidden, w->hq, w->hkv, w->ffn);
  if (w->d != 64 && w->d != 128) return fail(TREE_ERR_UNSUPPORTED, "tree_layer: head dim %d", w->d);
  if (w->hidden % 8 || w->ffn % 8) return fail(TREE_ERR_UNSUPPORTED, "tree_layer: hidden and ffn must be multiples of 8");
  if (!w->w_in || !w->wq || !w->wk || !w->wv || !w->wo || !w->w_post || !w->wgu || !w->wd)
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
  if ((rc = tree_gemm(xn, w->wq, q, nullptr, m, qd, w->hidden, TREE_GEMM_STORE, status, stream))) return rc;
  if ((rc = tree_gemm(xn, w->wk, kf, nullptr, m, kvd, w->hidden, TREE_GEMM_STORE, status, stream))) return rc;
  if ((rc = tree_gemm(xn, w->wv, vf, nullptr, m, kvd, w->hidden, TREE_GEMM_STORE, status, stream))) return rc;
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
