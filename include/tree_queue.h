/*
 * tree_queue.h -- host request planner: requests -> scheduling queue -> batches
 * laid out as prefix-tree forests for tree_pack_plan (tree_attn.h).
 *
 * Follows the basal-rs Architecture page:
 *   "01 / Request path: Validation and planning" -- a request's cost is the
 *       number of tokens to compute when shared prefixes are counted once;
 *   "01 / Request path: HRRN queue" -- the next request is the one with the
 *       highest (waiting time + estimated runtime) / estimated runtime;
 *       requests over long_tokens go to a separate long-request lane;
 *       schedule fifo restores arrival order;
 *   "01 / Request path: Batch and prefix tree" -- a batch is the first queued
 *       request and each subsequent one that fits within max_batch_tokens; its
 *       prompts are arranged into rows, each row a tree whose shared prompt
 *       prefixes are computed once; identical prompts share one readout;
 *   "04 / Scheduling" -- max_batch_tokens 8192, long_tokens 4096 (0 disables
 *       the lane); short batches go ahead of all long requests.
 *
 * Host only: nothing here touches the GPU.  The caller owns every array it
 * passes in (read during the call only); queues and batches are owned by the
 * library (tree_queue_destroy / tree_batch_free).  Status codes and
 * tree_last_error() are those of tree_attn.h.  Not thread-safe: one queue is
 * used by one thread at a time.
 */
#ifndef TREE_QUEUE_H
#define TREE_QUEUE_H

#include "tree_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One prompt block: its content key and its token count.  Blocks with equal
 * non-zero key and equal length hold the same tokens; key 0 = unique block
 * (never shared). */
typedef struct {
  uint64_t key;
  int32_t length; /* > 0 */
} tree_block_t;

/*
 * A request: its prompts, each a root-to-leaf path of blocks (template,
 * document/state, question, option order ...), and its questions, each read
 * out at the last tokens of two of its prompts (order 1 and order 2).
 */
typedef struct {
  int64_t id;                  /* caller's id, unique among queued requests */
  double arrival_ms;           /* arrival time on the caller's clock */
  int32_t n_prompts;           /* >= 1 */
  const int32_t *prompt_blocks; /* [n_prompts] blocks in each prompt, 1..max_depth */
  const tree_block_t *blocks;  /* the prompts' blocks, concatenated, root first */
  int32_t n_questions;         /* >= 0 */
  const int32_t *q_prompt1;    /* [n_questions] prompt whose last token reads out order 1 */
  const int32_t *q_prompt2;    /* [n_questions] ... order 2 */
} tree_request_t;

typedef struct {
  int32_t max_batch_tokens; /* cost limit of a batch of short requests */
  int32_t long_tokens;      /* requests costing more go to the long lane; 0 disables the lane */
  int32_t fifo;             /* 0: HRRN, 1: first in, first out */
  double ms_per_token;      /* estimated runtime per token to compute, > 0 */
  int32_t max_depth;        /* blocks on a prompt */
  int32_t max_row;          /* tokens in one row (tree) */
  int32_t n_resident;       /* root blocks whose K/V are resident (cost 0), e.g. the template */
  const uint64_t *resident_keys; /* [n_resident], copied at creation */
} tree_queue_opts_t;

/* The pages' defaults: 8192, 4096, HRRN, 0.01 ms per token, depth 8, row 32768, no resident keys. */
TREE_API int tree_queue_default_opts(tree_queue_opts_t *opts);

typedef struct tree_queue tree_queue_t;

TREE_API int tree_queue_create(const tree_queue_opts_t *opts, tree_queue_t **out);
TREE_API int tree_queue_destroy(tree_queue_t *q);

/*
 * Validate a request, compute its cost (tokens of its prompt tree, shared
 * prefixes once, resident roots free) and queue it in the short or the long
 * lane.  The request is copied.  Errors (nothing is queued): TREE_ERR_INVALID_ARG
 * (duplicate id, bad counts or indices, a question prompt that is a strict
 * prefix of another prompt of the request), TREE_ERR_BAD_TREE (length <= 0),
 * TREE_ERR_DEPTH, TREE_ERR_ROW_TOO_LONG (one prompt longer than max_row).
 */
TREE_API int tree_queue_push(tree_queue_t *q, const tree_request_t *req, int64_t *cost_out);

/* Drop a queued request (its client no longer waits); TREE_ERR_INVALID_ARG if not queued. */
TREE_API int tree_queue_cancel(tree_queue_t *q, int64_t id);

typedef struct {
  int32_t n_short, n_long; /* queued requests per lane */
} tree_queue_info_t;

TREE_API int tree_queue_info(const tree_queue_t *q, tree_queue_info_t *info);

typedef struct tree_batch tree_batch_t;

/*
 * Take the next batch at time now_ms.  Short lane first: its best request by
 * the schedule, then every other short request in schedule order whose
 * prompts fit -- the batch's cost (shared prefixes counted once across all its
 * requests) stays within max_batch_tokens, every row within max_row, at most
 * one resident root, and no question prompt of one request becomes a strict
 * prefix of a prompt of another.  With the short lane empty, the best long
 * request alone.  *out = NULL when both lanes are empty.  Taken requests leave
 * the queue.
 */
TREE_API int tree_queue_pop(tree_queue_t *q, double now_ms, tree_batch_t **out);

typedef struct {
  int32_t lane;                /* 0 short batch, 1 long request */
  int32_t n_requests;
  const int64_t *request_ids;  /* [n_requests] in the order taken */
  const int32_t *request_q0;   /* [n_requests + 1] each request's questions in spec.leaf1/leaf2 */
  int64_t cost;                /* tokens to compute */
  tree_spec_t spec;            /* the batch forest (blocks in first-seen order, parents first;
                                  identical blocks merged; questions in request order);
                                  arrays owned by the batch */
} tree_batch_view_t;

TREE_API int tree_batch_view(const tree_batch_t *b, tree_batch_view_t *view);
TREE_API int tree_batch_free(tree_batch_t *b);

#ifdef __cplusplus
}
#endif

#endif /* TREE_QUEUE_H */
