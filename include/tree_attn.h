/*
 * tree_attn.h -- C ABI of the packed prefix-tree attention library (GB300, sm_103a).
 *
 * The library computes the data-parallel hot path of a Llama forward over a
 * batch of prompts packed as prefix trees, as the basal-rs Architecture page
 * describes it:
 *
 *   tree_pack_plan  -- prompts -> per-row prefix trees -> one packed token row
 *                      ("01 / Request path: Batch and prefix tree";
 *                       "03 / Packing: Attention over tree blocks")
 *   tree_rope       -- rotary embedding at tree positions: a token's position
 *                      is its position in its own prompt ("03 / Packing")
 *   tree_attn_fwd   -- attention over tree blocks: a token sees the earlier
 *                      tokens of its own block and all tokens of its ancestor
 *                      blocks; sibling branches are masked ("03 / Packing";
 *                      f16 storage, f32 accumulation per "01 / Request path:
 *                      GPU forward pass")
 *   readout_decide  -- letter probabilities for both option orders, order 2
 *                      put back, averaged, calibrated with
 *                      p_cal = softmax(log(max(p, 1e-12)) / T)
 *                      ("02 / Basal protocol: Two option orders and calibration")
 *
 * Conventions for every call:
 *   - The return value is a status code (TREE_OK = 0 on success).  On failure
 *     tree_last_error() returns a message for the calling thread.
 *   - The caller owns all device memory; the library never allocates device
 *     memory, except tree_runtime_create, which allocates its buffers once
 *     and frees them in tree_runtime_destroy.  Plans live in host memory owned
 *     by the library (tree_pack_plan / tree_plan_free).
 *   - GPU work is enqueued on the caller's stream (NULL = legacy default
 *     stream) and never synchronised inside the library.  Launch errors are
 *     returned; errors found on the device (a bounded wait that gave up) are
 *     written to the caller's int32 `status` word in device memory, which the
 *     caller clears before the call and reads after synchronising.
 *   - f16 tensors are IEEE binary16, row-major, densely packed.
 */
#ifndef TREE_ATTN_H
#define TREE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TREE_API __attribute__((visibility("default")))
#else
#define TREE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st *tree_stream_t;

enum tree_status {
  TREE_OK = 0,
  TREE_ERR_INVALID_ARG = 1,   /* NULL pointer, bad size, question block not a leaf, ... */
  TREE_ERR_BAD_TREE = 2,      /* parent out of range, cycle, block length <= 0 */
  TREE_ERR_DEPTH = 3,         /* a tree deeper than max_depth blocks */
  TREE_ERR_ROW_TOO_LONG = 4,  /* a row (one tree) longer than max_row tokens */
  TREE_ERR_UNSUPPORTED = 5,   /* head dim not 64/128, hq % hkv != 0, misaligned pointer, > 255 letters */
  TREE_ERR_CUDA = 6,          /* a CUDA runtime call or launch failed */
  TREE_ERR_TIMEOUT = 7        /* written to `status` by a device wait that gave up */
};

/* Message describing the last error of the calling thread ("" if none). */
TREE_API const char *tree_last_error(void);

/* Library ABI version (major * 100 + minor). */
TREE_API int tree_version(void);

/* ------------------------------------------------------------------------ */
/* Planner (host only)                                                       */
/* ------------------------------------------------------------------------ */

/*
 * One batch as a forest of prompt blocks ("01 / Request path: Batch and prefix
 * tree": the prompts of a batch are arranged into rows, each row a tree whose
 * shared prefixes are computed once).
 *
 *   parent[b]   parent block of input block b, -1 for a root
 *   length[b]   tokens in block b, > 0
 *   key[b]      content key, NULL = every block unique.  Sibling blocks (same
 *               parent after merging) with equal non-zero key and equal
 *               length are one block: identical prompts share one block and
 *               one readout ("Batch and prefix tree").  Their children pool.
 *   resident[b] NULL = none.  1 = the block's K/V are already in the cache
 *               (e.g. the template, computed once at startup, "03 / Packing").
 *               Resident tokens must come first in the packed order.
 *   leaf1/leaf2 per question, the input blocks whose last token reads out the
 *               order-1 and order-2 letters; each must be a leaf after merging.
 * All arrays are host memory, read during the call only.
 */
typedef struct {
  int32_t n_blocks;
  const int32_t *parent;
  const int32_t *length;
  const uint64_t *key;
  const uint8_t *resident;
  int32_t n_questions;
  const int32_t *leaf1;
  const int32_t *leaf2;
} tree_spec_t;

/* Planner options; a zero field takes the default in brackets. */
typedef struct {
  int32_t max_fwd;   /* tokens per forward chunk, multiple of 128 [8192] */
  int32_t max_depth; /* blocks on a root-to-leaf path [8] */
  int32_t max_row;   /* tokens in one tree [32768] */
  int32_t tiling;    /* key tiles of the attention: 0 = 128 consecutive packed keys [0];
                        1 = by position: each query sees its keys in tiles of 128 positions of
                        its own prompt (key at position p in slot p % 128, tiles in increasing
                        position), so its result does not depend on the other prompts of the
                        batch ("05 / Reproducibility": attention tiled by position);
                        2 = gathered: the keys that some query of the tile sees, in packed
                        order, 128 to a tile (no tile spent on keys nobody in the query tile
                        sees: for batches of short prompts under a shared template) */
  int32_t pack_heads; /* q heads packed into one 128-row MMA tile with tiling 1 or 2 [1]: 1, 2, 4
                        or 8.  With R > 1 a query tile holds 256 / R tokens, attended as two MMA
                        tiles of R heads x 128 / R tokens that share each K/V tile; the attention
                        then needs hq / hkv == R.  With tiling 1 each query still takes its keys
                        in the same tiles, slots and order, so results stay batch-invariant. */
} tree_plan_opts_t;

typedef struct tree_plan tree_plan_t;

/*
 * Build a plan: merge identical sibling blocks, pack blocks in depth-first
 * pre-order (children in input order, roots in input order), give each token
 * its position in its own prompt and the end of its block's subtree, split the
 * forward tokens into chunks of max_fwd, list for every 128-row query tile the
 * 128-key tiles it sees (full or partial), and number the readout slots (the
 * last token of every leaf block, in packed order).
 *
 * Visibility in packed order: key j is visible to query i iff
 *     j <= i  and  i < send[j]
 * where send[j] is the end of the subtree of j's block.
 *
 * On success *out holds a new plan (free with tree_plan_free).  Errors:
 * TREE_ERR_INVALID_ARG, TREE_ERR_BAD_TREE, TREE_ERR_DEPTH,
 * TREE_ERR_ROW_TOO_LONG, TREE_ERR_UNSUPPORTED (max_fwd not a multiple of 128).
 */
TREE_API int tree_pack_plan(const tree_spec_t *spec, const tree_plan_opts_t *opts, tree_plan_t **out);

/*
 * Free a plan (NULL is accepted).  The largest host buffers of the plans freed
 * on a thread (device image, gathered keys, their run tables) are kept for the
 * next tree_pack_plan on that thread, so a caller planning batch after batch
 * does not pay for fresh memory each time; the thread holds at most the
 * buffers of the largest plan it has freed, released when it exits.
 */
TREE_API int tree_plan_free(tree_plan_t *plan);

typedef struct {
  int32_t n_input_blocks;
  int32_t n_blocks;      /* blocks after merging */
  int32_t n_tot;         /* packed tokens, resident included */
  int32_t n_res;         /* leading resident tokens */
  int32_t n_fwd;         /* n_tot - n_res: tokens whose Q/K/V the forward computes */
  int32_t n_chunks;
  int32_t n_qtiles;      /* over all chunks */
  int32_t n_entries;     /* (query tile, key tile) pairs that see anything */
  int32_t n_slots;       /* readout slots */
  int32_t n_questions;
  int32_t max_fwd;
  int32_t bm, bn;        /* query tile tokens (128; 256 / pack_heads with packed heads) / key tile rows (128) */
  int32_t max_pos;       /* 1 + largest position: rows needed in the RoPE table */
  int64_t pairs;         /* visible (query, key) pairs over all forward tokens */
  size_t dev_bytes;      /* size of the device image (tree_plan_upload) */
  /* byte offsets of the device image's arrays (int32 each) */
  size_t off_pos, off_send, off_qtile, off_ent, off_order, off_chunk, off_slot_tok, off_r1, off_r2;
  size_t off_runs;       /* run tables of the key tiles (see tree_plan_host_view_t.runs) */
  int32_t tiling;        /* as in tree_plan_opts_t */
  size_t off_vkeys, off_vruns; /* tiling 1, 2: per entry its 128 gathered keys and its run table */
  int32_t pack_heads;    /* as in tree_plan_opts_t (1 when not packed) */
} tree_plan_info_t;

TREE_API int tree_plan_query(const tree_plan_t *plan, tree_plan_info_t *info);

typedef struct {
  int32_t q0, q1;        /* packed token range of the chunk's queries */
  int32_t t0, t1;        /* its query tiles */
  int64_t pairs;         /* visible pairs of its queries */
  int32_t n_entries;     /* tile pairs the kernel visits */
} tree_chunk_info_t;

TREE_API int tree_plan_chunk(const tree_plan_t *plan, int32_t chunk, tree_chunk_info_t *info);

/*
 * Read-only host view of the plan's tables (valid until tree_plan_free).
 * Blocks are in packed order.  ent[e] = (key_tile << 1) | partial.
 */
typedef struct {
  const int32_t *block_map;                       /* [n_input_blocks] input block -> packed block */
  const int32_t *blk_start, *blk_len, *blk_parent, *blk_depth, *blk_pos0, *blk_send, *blk_resident,
      *blk_slot;                                  /* [n_blocks] */
  const int32_t *pos;                             /* [n_tot] */
  const int32_t *send;                            /* [ceil(n_tot/128)*128], 0 past n_tot */
  const int32_t *chunk_q0, *chunk_q1, *chunk_t0, *chunk_t1; /* [n_chunks] */
  const int32_t *qt_row0, *qt_row1, *qt_ent0, *qt_ent1;     /* [n_qtiles] */
  const int32_t *ent;                             /* [n_entries] */
  const int32_t *qt_order;                        /* [n_qtiles] per chunk, most entries first */
  const int32_t *slot_tok;                        /* [n_slots] */
  const int32_t *r1, *r2;                         /* [n_questions] readout slots of each question */
  const void *image;                              /* the device image, host copy */
  size_t image_bytes;
  const int32_t *runs;  /* [ceil(n_tot/128)][84] per 128-key tile, its keys split into maximal runs of
                           equal send: word 0 the number of runs n; if n <= 16, words 4 + r the run's
                           send, words 20 + 4r .. 23 + 4r its keys as a 128-bit mask (key c of the
                           tile is bit c % 32 of word c / 32); all else 0.  A query i sees the keys
                           of run r, apart from keys after i, iff i < send of r. */
  /* tiling 1 and 2 (else NULL).  Entry e of the tile lists is a virtual key tile.  ent[e] =
     (e << 2) | contiguous << 1 | 1 (contiguous: its slots hold the consecutive packed keys
     vkeys[128 e] + c), or (j0 << 2) | 2 when every row of the query tile takes this range from it
     and sees every slot, slot c holding key j0 + c (no mask: a packed key tile).  Per entry: vkeys[128 e + c] = the packed key in slot c (0 for an empty slot, which no query
     sees); vruns[72 e ..]: word 0 the number of runs n (<= 16), words 4-7 the 128-bit mask of
     the query tile's rows that take their keys of this position range from this entry, then per
     run r words 8 + 4r .. 11 + 4r = {first slot c0, last slot c1, packed key j0 in c0, its send}:
     the run's slots hold the consecutive keys j0 + (c - c0) of one block.  Query i of an
     assigned row sees slot c of run r iff c - c0 <= i - j0 and j0 <= i < send.  With tiling 2
     every row of the query tile is assigned to every entry of its list, an entry holds at most
     16 runs, and "contiguous" means that all 128 slots hold consecutive keys (it may have
     several runs). */
  const int32_t *vkeys, *vruns;
} tree_plan_host_view_t;

TREE_API int tree_plan_tables(const tree_plan_t *plan, tree_plan_host_view_t *view);

/*
 * Copy the plan's device image (info.dev_bytes bytes) into caller-owned device
 * memory `dev_buf` (16-byte aligned, `bytes` >= dev_bytes) on `stream`.  The
 * host copy is pageable; the plan may be freed once this returns.
 */
TREE_API int tree_plan_upload(const tree_plan_t *plan, void *dev_buf, size_t bytes, tree_stream_t stream);

/*
 * tree_plan_upload through caller-owned page-locked host memory, for callers
 * that plan the next batch while the GPU still runs the current one.  A copy
 * from pageable memory goes through the driver's staging buffers and can hold
 * the calling thread until the GPU has drained earlier work; this call copies
 * the image into `host_staging` (page-locked, e.g. cudaHostAlloc,
 * `staging_bytes` >= dev_bytes) on the calling thread and then enqueues an
 * asynchronous host-to-device copy from it on `stream`, so it never waits for
 * the GPU.  Upload into a device buffer that no queued kernel still reads
 * (e.g. two buffers used in turn) on a copy stream, and make the compute
 * stream wait for that copy (an event) before its launches.
 *
 * Ownership: `host_staging` stays the caller's; it must not be rewritten or
 * freed until the copy has executed on `stream` (record an event after this
 * call and wait on it first).  The plan may be freed once this returns.
 * Errors: TREE_ERR_INVALID_ARG (NULL pointer, buffer too small),
 * TREE_ERR_UNSUPPORTED (dev_buf not 16-byte aligned), TREE_ERR_CUDA.
 * This is plumbing around the planner; the pages define no such call.
 */
TREE_API int tree_plan_upload_staged(const tree_plan_t *plan, void *dev_buf, size_t bytes, void *host_staging,
                                     size_t staging_bytes, tree_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Rotary embedding at tree positions                                        */
/* ------------------------------------------------------------------------ */

/*
 * Fill host_out[max_pos][d/2][2] with {cos, sin} of pos * theta^(-2i/d),
 * evaluated in double and rounded to float (the table form of the AstrAI
 * inference page, "Rotary Embedding Backend").  d even, max_pos > 0.
 */
TREE_API int tree_rope_table(float *host_out, int32_t max_pos, int32_t d, double theta);

/*
 * Rotate, in place, the queries and keys of forward chunk `chunk`, pair
 * (i, i + d/2) by the angle of the token's tree position (plan pos table):
 *
 *   q   f16 [q1-q0, hq, d]   the chunk's query rows (row r = packed token q0 + r)
 *   k   f16 [n_tot, hkv, d]  the whole KV space; rows [q0, q1) are rotated
 *   cos_sin  f32 [max_pos][d/2][2] device table from tree_rope_table,
 *            max_pos >= info.max_pos
 *
 * Arithmetic in f32 (y_i = fma(x_i, cos, -(x_{i+d/2} sin)), y_{i+d/2} =
 * fma(x_{i+d/2}, cos, x_i sin)), stored f16 (round to nearest even).  plan_dev
 * is the device image from tree_plan_upload.  d a multiple of 16 and <= 256;
 * q and k 16-byte aligned.  q may be NULL (hq is then ignored): only the keys
 * are rotated, for a caller that has rotated its queries elsewhere.
 * `status` (device int32, may be NULL) is the status word of the other
 * kernels; this kernel never waits and never writes it.
 */
TREE_API int tree_rope(const tree_plan_t *plan, const void *plan_dev, int32_t chunk, void *q, void *k,
              int32_t hq, int32_t hkv, int32_t d, const float *cos_sin, int32_t max_pos,
              int32_t *status, tree_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Attention over tree blocks                                                */
/* ------------------------------------------------------------------------ */

typedef struct {
  int32_t hq, hkv, d;  /* query heads, kv heads (hq % hkv == 0, q head h reads kv head h/(hq/hkv)), d in {64,128} */
  float scale;         /* scores are q.k * scale; 0 = 1/sqrt(d) (AstrAI inference page, "KV Cache") */
  int32_t *work;       /* device int32[2], or NULL.  Work counter of the persistent CTAs: when given,
                          CTAs take (query tile, kv head) items in longest-first order as they free
                          up; it must hold {0, 0} before the first call and each call leaves it at
                          {0, 0} (the last CTA resets it), so calls on one stream can reuse it;
                          calls that may overlap on the GPU need separate counters.  NULL: each CTA
                          takes a fixed round-robin share of the items (no scratch memory). */
  int32_t self_test;   /* 0 normally.  Nonzero: a self-test of the device-side failure detection;
                          before issuing any copy or MMA each CTA waits on a barrier that nothing
                          arrives on, gives up after 2 ms, writes TREE_ERR_TIMEOUT to `status`, and
                          winds down; no output is written.  The context stays usable. */
} tree_attn_params_t;

/*
 * Attention of forward chunk `chunk` over tree blocks:
 *
 *   O[i, h] = sum_{j visible to i} softmax_j(scale * Q[i,h] . K[j,g]) V[j,g],
 *   g = h / (hq/hkv), visible = j <= i and i < send[j]
 *
 *   q    f16 [q1-q0, hq, d]   post-RoPE queries of the chunk
 *   k, v f16 [n_tot, hkv, d]  post-RoPE keys and values of the whole KV space
 *                             (resident tokens, earlier chunks and this chunk)
 *   o    f16 [q1-q0, hq, d]   output, normalised
 *   lse  f32 [q1-q0, hq] or NULL: natural-log sum of exp of the scaled scores
 *
 * Scores, softmax and accumulation in f32; probabilities rounded to f16 for
 * the P.V product.  All tensors 16-byte aligned.  `status` (device int32, may
 * be NULL) receives TREE_ERR_TIMEOUT if a pipeline wait gave up.
 */
TREE_API int tree_attn_fwd(const tree_plan_t *plan, const void *plan_dev, int32_t chunk, const void *q,
                  const void *k, const void *v, void *o, float *lse, const tree_attn_params_t *params,
                  int32_t *status, tree_stream_t stream);

/*
 * tree_attn_fwd_noalloc -- the same attention for callers that cannot
 * allocate device memory: a host program linking only this library with no
 * allocator of its own, or code whose device memory belongs to another
 * runtime's pool, where a private cudaMalloc would bypass that runtime's
 * accounting and synchronise the device.  The pages that define the method
 * have no counterpart to this entry point: it only changes where scratch lives.
 *
 * Arguments and results are those of tree_attn_fwd except that params->work
 * must be NULL: the persistent CTAs' work counters live in a device array
 * inside the library, one pair per chunk index, at most 256 chunks per plan
 * (TREE_ERR_UNSUPPORTED beyond that).  The array (2 KB) stays resident on
 * every device that has loaded the library until the process exits.  Each
 * call clears its chunk's counter on `stream` before the launch.  Calls for
 * the same chunk index that may run at the same time on the GPU (different
 * streams, several plans) share that counter and race: serialise them.
 * The first call on each device (and the first after that device's context
 * has been replaced, by cudaDeviceReset for instance) looks up the array's
 * device address; make that first call before any stream capture begins.
 * Nothing is allocated.
 */
TREE_API int tree_attn_fwd_noalloc(const tree_plan_t *plan, const void *plan_dev, int32_t chunk, const void *q,
                                   const void *k, const void *v, void *o, float *lse,
                                   const tree_attn_params_t *params, int32_t *status, tree_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Rows over several GPUs (host only)                                        */
/* ------------------------------------------------------------------------ */

/*
 * Rows of one batch shared out over n_ranks GPUs.  A query sees only its own
 * prompt ("01 / Request path: Batch and prefix tree"; "03 / Packing: Attention
 * over tree blocks"), so each GPU can plan and run a share of the rows with no
 * data exchanged; every GPU keeps the resident blocks (the template, "03 /
 * Packing: Shared state computed once"), and decisions are gathered on the host.
 *
 * A row is the subtree of a non-resident block whose parent is resident or
 * absent, after identical siblings merge (rows that merge stay one).  Rows
 * joined by a question (its two leaves in different rows) form one unit.  A
 * unit costs its visible (query, key) pairs per head (a query at position p
 * sees p + 1 keys).  Units are assigned longest first (ties: first in packed
 * order) to the rank with the least cost so far (ties: lowest rank).
 *
 *   spec, opts     the batch, as for tree_pack_plan (opts->tiling is ignored)
 *   block_rank     out, host int32 [spec->n_blocks]: the rank of every input
 *                  block, -1 for resident blocks (kept by every rank)
 *   question_rank  out, host int32 [spec->n_questions]: the rank answering it
 *   rank_pairs     out, host int64 [n_ranks] or NULL: visible pairs per head
 * Errors: those of tree_pack_plan; TREE_ERR_INVALID_ARG for n_ranks < 1 or a
 * question whose leaf is a resident block.
 */
TREE_API int tree_shard_rows(const tree_spec_t *spec, const tree_plan_opts_t *opts, int32_t n_ranks,
                             int32_t *block_rank, int32_t *question_rank, int64_t *rank_pairs);

/* One rank's share of a batch, written by tree_shard_select into caller arrays
 * of (at least) spec->n_blocks and spec->n_questions entries. */
typedef struct {
  int32_t n_blocks;         /* out: blocks kept, in input order */
  int32_t *parent;          /* [n_blocks] parent among the kept blocks, -1 for a root */
  int32_t *length;          /* [n_blocks] */
  uint64_t *key;            /* [n_blocks] or NULL; 0 where the spec has no keys */
  uint8_t *resident;        /* [n_blocks] or NULL; 0 where the spec has none */
  int32_t *block_index;     /* [n_blocks] input block of each kept block */
  int32_t n_questions;      /* out: questions kept, in input order */
  int32_t *leaf1, *leaf2;   /* [n_questions] their leaves among the kept blocks */
  int32_t *question_index;  /* [n_questions] input question of each kept one */
} tree_shard_t;

/*
 * The blocks and questions of `rank` (as tree_shard_rows assigned them) as a
 * forest of their own, blocks and questions in input order: planning it packs
 * the rank's rows in the same order as in the whole batch.  Host only.
 * Errors: TREE_ERR_INVALID_ARG (NULL arrays; a kept block whose parent is not
 * kept; a question whose leaves are not kept).
 */
TREE_API int tree_shard_select(const tree_spec_t *spec, const int32_t *block_rank, const int32_t *question_rank,
                               int32_t rank, tree_shard_t *out);

/* ------------------------------------------------------------------------ */
/* Letter readout and calibration                                            */
/* ------------------------------------------------------------------------ */

/*
 * For each question q (one warp per question):
 *   l1 = logits[r1[q], 0:n], l2 = logits[r2[q], 0:n], n = n_letters[q] in 1..255
 *   p     = (softmax(l1) + reverse(softmax(l2))) / 2       reverse: k -> n-1-k
 *   p_cal = softmax(log(max(p, 1e-12)) / T[q])             T[q] > 0
 *   choice[q] = argmax p_cal (lowest index on ties), taken as argmax of p
 *
 *   logits      f32 [n_slots, stride] device
 *   r1, r2, n_letters  int32 [n_q] device;  temperature f32 [n_q] device
 *   p_cal       f32 [n_q, stride] device, zero past n
 *   p_avg       f32 [n_q, stride] device or NULL, zero past n
 *   choice      int32 [n_q] device or NULL
 *   status      device int32 or NULL: TREE_ERR_INVALID_ARG if some n is out
 *               of 1..min(stride,255) or some T <= 0 (that question's
 *               outputs are zero, choice -1)
 * All arithmetic in f32.  n_q == 0 is a no-op.
 * The kernel is a programmatic dependent launch: for strides up to 32 it reads
 * r1, r2, n_letters and temperature before the kernel ahead of it in the
 * stream has finished (the logits only after), so a kernel that lets its
 * dependents launch early (griddepcontrol.launch_dependents) must not write
 * them; the library's own kernels never do.
 */
TREE_API int readout_decide(const float *logits, int32_t stride, const int32_t *r1, const int32_t *r2,
                   const int32_t *n_letters, const float *temperature, int32_t n_q, float *p_cal,
                   float *p_avg, int32_t *choice, int32_t *status, tree_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Runtime: the whole path of one batch per call                             */
/* ------------------------------------------------------------------------ */

/*
 * For callers that run batch after batch on one stream: tree_runtime_step
 * plans the batch and enqueues the plan image's transfer, tree_rope and
 * tree_attn_fwd for every chunk, and readout_decide, as one chain of kernels
 * (each overlapping its predecessor's tail and waiting for it before reading
 * its results).  The runtime owns two device plan buffers and two page-locked
 * staging buffers used in turn, so the host can plan the next batch while the
 * GPU runs this one, plus the attention work counters.  This is orchestration
 * of the calls above; the pages define no such call.
 *
 * tree_runtime_create allocates, once: 2 x max_plan_bytes of device memory and
 * of page-locked host memory, and 8 x max_chunks bytes of device counters (it
 * synchronises the device).  tree_runtime_destroy waits for the device and
 * frees them.  A runtime serves one stream at a time (steps on different
 * streams would share its buffers and race).
 */
typedef struct tree_runtime tree_runtime_t;

TREE_API int tree_runtime_create(size_t max_plan_bytes, int32_t max_chunks, tree_runtime_t **out);
TREE_API int tree_runtime_destroy(tree_runtime_t *rt);

typedef struct {
  const tree_spec_t *spec;        /* the batch (host memory, read during the call) */
  const tree_plan_opts_t *opts;   /* may be NULL: defaults */
  void *q;                        /* f16 [n_fwd, hq, d]: pre-RoPE queries of all chunks, rotated in place */
  void *k;                        /* f16 [n_tot, hkv, d]: keys, forward rows rotated in place */
  const void *v;                  /* f16 [n_tot, hkv, d] */
  void *o;                        /* f16 [n_fwd, hq, d] output */
  float *lse;                     /* f32 [n_fwd, hq] or NULL */
  const float *cos_sin;           /* tree_rope_table on the device */
  int32_t max_pos;                /* rows of cos_sin, >= the plan's max_pos */
  int32_t hq, hkv, d;
  float scale;                    /* 0 = 1/sqrt(d) */
  const float *logits;            /* f32 [n_slots, stride]; the readout arguments may be NULL  */
  int32_t stride;                 /*   when the batch has no questions                          */
  const int32_t *n_letters;       /* [n_questions] */
  const float *temperature;       /* [n_questions] */
  float *p_cal, *p_avg;           /* [n_questions, stride]; p_avg may be NULL */
  int32_t *choice;                /* [n_questions] or NULL */
  int32_t *status;                /* device int32 or NULL (as for the calls above) */
  void *attn_events[2];           /* cudaEvent_t pair or NULLs: recorded on the stream just before the
                                     first and just after the last tree_attn_fwd launch of the step */
} tree_step_args_t;

/*
 * One batch.  Errors: those of the calls above, TREE_ERR_UNSUPPORTED when the
 * plan image exceeds max_plan_bytes or the plan has more chunks than
 * max_chunks.  info_out (may be NULL) receives the batch's plan summary.
 */
TREE_API int tree_runtime_step(tree_runtime_t *rt, const tree_step_args_t *args, tree_plan_info_t *info_out,
                               tree_stream_t stream);

/*
 * Host-buffer steps.  tree_runtime_attach_io gives the runtime two device sets
 * of input and output buffers sized by `caps`, a copy stream of its own and
 * the events that order them (it synchronises the device; calling it again
 * replaces the sets).  tree_runtime_step_host then takes one batch whose
 * inputs and outputs live in HOST memory:
 *
 *   copy stream:  wait until the step two calls back has finished with set b
 *                 (b alternates), then q, k, v, logits, n_letters, temperature
 *                 host -> set b (one cudaMemcpyAsync each)
 *   stream:       wait for those copies, tree_runtime_step on set b, then the
 *                 decisions (choice, p_cal, p_avg) and o, where the caller
 *                 passes host buffers for them, device -> host
 *
 * so the upload of batch s+1 runs while batch s computes when the caller
 * issues step s+1 before synchronising on `stream`.  The call returns once the
 * work is enqueued: the host outputs are valid after `stream` has completed
 * the step, and the host inputs may be rewritten once the step has reached
 * `stream` (the copies of step s run before step s's compute starts).  Host
 * buffers should be page-locked; pageable ones work but their copies do not
 * overlap.  Resident key rows arrive with the keys as they are (already
 * rotated, as for tree_runtime_step).  Errors: TREE_ERR_INVALID_ARG (no
 * buffers attached, NULL inputs, sizes above caps or heads/d/stride different
 * from caps), those of tree_runtime_step.
 */
typedef struct {
  int32_t max_fwd;       /* forward (query) rows per batch */
  int32_t max_tot;       /* key rows per batch (resident + forward) */
  int32_t hq, hkv, d;    /* heads and head dimension of every step */
  int32_t stride;        /* letters per logits row; 0 = no readout buffers */
  int32_t max_slots;     /* readout slots (logits rows) per batch */
  int32_t max_questions; /* questions per batch */
} tree_io_caps_t;

TREE_API int tree_runtime_attach_io(tree_runtime_t *rt, const tree_io_caps_t *caps);

typedef struct {
  const tree_spec_t *spec;        /* the batch (host memory, read during the call) */
  const tree_plan_opts_t *opts;   /* may be NULL: defaults */
  const void *q;                  /* host f16 [n_fwd, hq, d] pre-RoPE queries */
  const void *k;                  /* host f16 [n_tot, hkv, d] keys (resident rows rotated) */
  const void *v;                  /* host f16 [n_tot, hkv, d] */
  void *o;                        /* host f16 [n_fwd, hq, d] output, or NULL: not copied back */
  const float *cos_sin;           /* tree_rope_table on the device */
  int32_t max_pos;
  float scale;                    /* 0 = 1/sqrt(d) */
  const float *logits;            /* host f32 [n_slots, stride]; the readout arguments may be NULL */
  const int32_t *n_letters;       /*   when the batch has no questions: host [n_questions]        */
  const float *temperature;       /* host [n_questions] */
  float *p_cal, *p_avg;           /* host [n_questions, stride]; either may be NULL: not copied back */
  int32_t *choice;                /* host [n_questions] or NULL */
  int32_t *status;                /* device int32 or NULL */
} tree_host_step_args_t;

TREE_API int tree_runtime_step_host(tree_runtime_t *rt, const tree_host_step_args_t *args,
                                    tree_plan_info_t *info_out, tree_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TREE_ATTN_H */
