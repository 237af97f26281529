/*
 * tree_layer.h -- the Llama layer around the tree attention (GB300, sm_103a):
 * the projections as tensor-core GEMMs with fused epilogues, and RMSNorm.
 *
 * The basal-rs Architecture page ("01 / Request path: GPU forward pass") runs
 * the Llama model in f16 over the batch as one compact token list, without
 * padding.  A layer over the packed tokens of a batch is
 *
 *     xn = rmsnorm(x, w_in)                      tree_rmsnorm
 *     q, k, v = xn [Wq; Wk; Wv]^T               tree_gemm_qkv (k, v into the cache rows)
 *     q, k rotated at tree positions             tree_rope           (tree_attn.h)
 *     o = attention over tree blocks             tree_attn_fwd       (tree_attn.h)
 *     h = x + o Wo^T                             tree_gemm RESIDUAL
 *     hn = rmsnorm(h, w_post)                    tree_rmsnorm
 *     g = silu(hn Wg^T) * (hn Wu^T)              tree_gemm SWIGLU
 *     y = h + g Wd^T                             tree_gemm RESIDUAL
 *
 * Conventions as in tree_attn.h: status codes, caller-owned device memory,
 * work enqueued on the caller's stream (launched so that it may overlap the
 * tail of the kernel before it; it waits for that kernel before reading).
 * f16 tensors are row-major, densely packed, 16-byte aligned.
 */
#ifndef TREE_LAYER_H
#define TREE_LAYER_H

#include "tree_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

enum tree_gemm_epilogue {
  TREE_GEMM_STORE = 0,    /* C = A B^T */
  TREE_GEMM_RESIDUAL = 1, /* C = A B^T + R   (R [m, n], may be C itself) */
  TREE_GEMM_SWIGLU = 2,   /* C = silu(A G^T) * (A U^T), B = [G; U] with 2n rows, silu(g) = g / (1 + e^-g) */
  TREE_GEMM_STORE_F32 = 3 /* C = A B^T as f32 (C is float [m, n]) */
};

/*
 * C[m, n] = epilogue(A B^T): A f16 [m, k] (an activation), B f16 [n, k] (a
 * Linear weight, [2n, k] for SWIGLU), f32 accumulation over the whole of k in
 * one fixed order (no split over k), the epilogue in f32, C f16 [m, n]
 * (f32 for STORE_F32).
 * n and k multiples of 8; m >= 0 (0: nothing to do).  `status` (device int32,
 * may be NULL) receives TREE_ERR_TIMEOUT if a bounded device wait gives up.
 * Errors: TREE_ERR_INVALID_ARG (NULL, sizes, unknown epilogue, RESIDUAL without
 * R), TREE_ERR_UNSUPPORTED (n or k not a multiple of 8, misaligned pointer),
 * TREE_ERR_CUDA.
 */
TREE_API int tree_gemm(const void *a, const void *b, void *c, const void *r, int32_t m, int32_t n, int32_t k,
                       int32_t epi, int32_t *status, tree_stream_t stream);

/*
 * tree_gemm with the output tile width chosen by the caller: tile_n 256 (wide
 * tiles, for large m), 64 (narrow tiles: more of them, so a small m still
 * spreads the weight reads over every SM), or 0 (tree_gemm's choice: narrow
 * for m <= 384, except with the SwiGLU epilogue, else wide).  The width changes
 * only the speed: every output is the same f32 sum over k in the same order.
 */
TREE_API int tree_gemm_ex(const void *a, const void *b, void *c, const void *r, int32_t m, int32_t n, int32_t k,
                          int32_t epi, int32_t tile_n, int32_t *status, tree_stream_t stream);

/*
 * The three projections of the attention block in one GEMM: W = [Wq; Wk; Wv]
 * f16 [nq + 2 nkv, k]; the output columns go to q f16 [m, nq], k and v f16
 * [m, nkv] (e.g. the forward rows of the caches).  Each output is the same f32
 * sum as tree_gemm's.  nq, nkv, k multiples of 8.
 */
TREE_API int tree_gemm_qkv(const void *a, const void *wqkv, void *q, void *k, void *v, int32_t m, int32_t nq,
                           int32_t nkv, int32_t kdim, int32_t *status, tree_stream_t stream);

/*
 * y[i, :] = f16( f16(x[i, :] / sqrt(mean_j x[i, j]^2 + eps)) * w ), the Llama
 * RMSNorm with its f32 statistics: the normalised row is rounded to f16 before
 * the f16 weight multiplies it.  x, y f16 [rows, cols] (y may be x), w f16
 * [cols]; cols a multiple of 8 and at most 16384.
 */
TREE_API int tree_rmsnorm(const void *x, const void *w, void *y, int32_t rows, int32_t cols, float eps,
                          tree_stream_t stream);

/* The weights of one Llama layer (device f16, row-major, 16-byte aligned). */
typedef struct {
  int32_t hidden, hq, hkv, d, ffn; /* model width, query / kv heads, head dim (64 or 128), MLP width */
  float eps;                       /* RMSNorm epsilon (Llama: 1e-5) */
  const void *w_in;                /* [hidden]            RMSNorm before attention */
  const void *wqkv;                /* [(hq + 2 hkv) d, hidden]: the q rows, then the k rows, then the v rows */
  const void *wo;                  /* [hidden, hq * d] */
  const void *w_post;              /* [hidden]            RMSNorm before the MLP */
  const void *wgu;                 /* [2 * ffn, hidden]   gate rows, then up rows */
  const void *wd;                  /* [hidden, ffn] */
} tree_layer_weights_t;

/* Bytes of the workspace tree_layer_fwd needs for this plan and these sizes. */
TREE_API int tree_layer_workspace_bytes(const tree_plan_t *plan, const tree_layer_weights_t *w, size_t *bytes);

/*
 * One Llama layer over the forward tokens of a planned batch (the sequence at
 * the top of this header), every chunk of the plan:
 *
 *   x        f16 [n_fwd, hidden]   the forward tokens' hidden states, packed order
 *   k_cache, v_cache f16 [n_tot, hkv * d]  rows [0, n_res) hold the resident
 *            tokens' post-RoPE keys and their values (read); rows [n_res, n_tot)
 *            receive this layer's post-RoPE keys and values
 *   y        f16 [n_fwd, hidden]   the layer's output (may not alias x)
 *   cos_sin  f32 rotary table (tree_rope_table), max_pos >= info.max_pos
 *   workspace  device memory of tree_layer_workspace_bytes, 256-byte aligned
 *   work     device int32 [2 * n_chunks] attention work counters, {0} before the
 *            first call (each call leaves them 0), or NULL
 *
 * All launches go to `stream` in order; nothing is synchronised.  Errors as the
 * calls it makes, plus TREE_ERR_INVALID_ARG for a short workspace.
 */
TREE_API int tree_layer_fwd(const tree_plan_t *plan, const void *plan_dev, const tree_layer_weights_t *w,
                            const void *x, void *k_cache, void *v_cache, void *y, const float *cos_sin,
                            int32_t max_pos, void *workspace, size_t workspace_bytes, int32_t *work,
                            int32_t *status, tree_stream_t stream);

/*
 * The final layer with its pruning ("01 / Request path: GPU forward pass": in
 * the final layer the MLP block and the logits are computed only for readout
 * positions and answer letters).  The attention block runs over every forward
 * token (their keys and values are written as in tree_layer_fwd); then only the
 * plan's readout slots (the last token of each leaf) continue:
 *
 *   h_s = x_s + o_s Wo^T;  y_s = h_s + (silu(hn_s Wg^T) * (hn_s Wu^T)) Wd^T
 *   logits = rmsnorm(y_s, w_final) W_letters^T       (f32, [n_slots, stride])
 *
 *   w_final    f16 [hidden]          the model's final RMSNorm
 *   w_letters  f16 [stride, hidden]  the LM-head rows of the answer letters, gathered once
 *                                    by the caller (row l = letter l; unused rows may be 0)
 *   stride     letters per logits row, a multiple of 8 (the readout_decide stride)
 *   logits     f32 [n_slots, stride] feeds readout_decide with the plan's r1/r2
 *
 * Every readout slot must be a forward token (TREE_ERR_INVALID_ARG otherwise).
 */
TREE_API int tree_last_layer_workspace_bytes(const tree_plan_t *plan, const tree_layer_weights_t *w, size_t *bytes);

TREE_API int tree_last_layer_fwd(const tree_plan_t *plan, const void *plan_dev, const tree_layer_weights_t *w,
                                 const void *x, void *k_cache, void *v_cache, const float *cos_sin, int32_t max_pos,
                                 const void *w_final, const void *w_letters, int32_t stride, float *logits,
                                 void *workspace, size_t workspace_bytes, int32_t *work, int32_t *status,
                                 tree_stream_t stream);

/*
 * A whole decision forward: n_layers Llama layers over the planned batch, the
 * last one pruned to the readout rows, ending in the letter logits
 * (readout_decide then takes them with the plan's r1 / r2).
 *
 *   layers    [n_layers] weights, host array of device pointers (layer l reads layers[l])
 *   x         f16 [n_fwd, hidden] the forward tokens' input hidden states (embeddings)
 *   k_caches, v_caches  host arrays [n_layers] of f16 [n_tot, hkv * d] caches (as in tree_layer_fwd)
 *   workspace tree_model_workspace_bytes bytes, 256-byte aligned
 * Every layer must have the same sizes.  Launches only; nothing is synchronised.
 */
TREE_API int tree_model_workspace_bytes(const tree_plan_t *plan, const tree_layer_weights_t *w, size_t *bytes);

TREE_API int tree_model_fwd(const tree_plan_t *plan, const void *plan_dev, const tree_layer_weights_t *layers,
                            int32_t n_layers, const void *x, void *const *k_caches, void *const *v_caches,
                            const float *cos_sin, int32_t max_pos, const void *w_final, const void *w_letters,
                            int32_t stride, float *logits, void *workspace, size_t workspace_bytes, int32_t *work,
                            int32_t *status, tree_stream_t stream);

/*
 * Long-request lane ("04 / Scheduling": a request over long_tokens runs in its
 * own lane that shares the GPU with short batches and yields it between layers:
 * after a layer, if it has run for at least long_slice_ms, it gives the GPU back
 * and later resumes at the next layer with the same tensors).
 *
 * A session is tree_model_fwd cut at layer boundaries.  It keeps the caller's
 * buffers (arguments as tree_model_fwd; they must stay valid and untouched
 * until the session is done) and the next layer to run; the plan is built once
 * and serves every layer.  tree_session_run enqueues whole layers on `stream`,
 * waiting for each layer's end (an event), until the wall time since the call
 * began reaches slice_ms or the last layer (with the logits) is done.  It always
 * runs at least one layer.  The results equal tree_model_fwd's bit for bit,
 * however the layers are cut into slices and whatever runs on the GPU between
 * slices.
 */
typedef struct tree_session tree_session_t;

TREE_API int tree_session_create(const tree_plan_t *plan, const void *plan_dev, const tree_layer_weights_t *layers,
                                 int32_t n_layers, const void *x, void *const *k_caches, void *const *v_caches,
                                 const float *cos_sin, int32_t max_pos, const void *w_final, const void *w_letters,
                                 int32_t stride, float *logits, void *workspace, size_t workspace_bytes,
                                 int32_t *work, int32_t *status, tree_session_t **out);

/* *layers_run = layers this call ran; *done = 1 once the last layer has run. */
TREE_API int tree_session_run(tree_session_t *s, double slice_ms, tree_stream_t stream, int32_t *layers_run,
                              int32_t *done);

TREE_API int tree_session_destroy(tree_session_t *s);

#ifdef __cplusplus
}
#endif

#endif /* TREE_LAYER_H */
