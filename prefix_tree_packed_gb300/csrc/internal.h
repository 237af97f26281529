// Internal declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "tree_attn.h"

namespace tree {

// Record a message for tree_last_error() and return `code`.
int fail(int code, const char *fmt, ...);
// Record success (clears nothing; returns TREE_OK).
inline int ok() { return TREE_OK; }

// Host plan: every table as int32 vectors plus the device image.
struct Plan {
  int32_t n_input_blocks = 0, n_blocks = 0, n_tot = 0, n_res = 0, n_chunks = 0;
  int32_t max_fwd = 8192, bm = 128, bn = 128, max_pos = 0, n_questions = 0;
  int64_t pairs = 0;
  std::vector<int32_t> block_map;
  std::vector<int32_t> blk_start, blk_len, blk_parent, blk_depth, blk_pos0, blk_send, blk_resident,
      blk_slot;
  // pos [n_tot] and send [ceil(n_tot/128)*128] live inside the device image
  std::vector<int32_t> chunk_q0, chunk_q1, chunk_t0, chunk_t1, chunk_nent;
  std::vector<int64_t> chunk_pairs;
  std::vector<int32_t> qt_row0, qt_row1, qt_ent0, qt_ent1, ent, qt_order;
  std::vector<int32_t> slot_tok, r1, r2;
  // device image: int32 words, arrays 16-byte aligned
  std::vector<int32_t> image;
  size_t off_pos = 0, off_send = 0, off_qtile = 0, off_ent = 0, off_order = 0, off_chunk = 0,
         off_slot_tok = 0, off_r1 = 0, off_r2 = 0, off_runs = 0;  // in int32 words
  // tiling by position: per entry its gathered keys and run table (see tree_plan_host_view_t)
  int32_t tiling = 0;
  int32_t pack_heads = 1;  // q heads per 128-row MMA tile (1: one head per tile)
  std::vector<int32_t> vkeys, vruns;
  size_t off_vkeys = 0, off_vruns = 0;
};

// Run table of a 128-key tile, in the device image (kRunWords int32 words per
// key tile): the tile's keys split into maximal runs of equal subtree end.
// A query i sees the keys of run r (apart from keys after i) iff i < end[r],
// so its 128-bit visibility mask is the OR of those runs' masks.
//   word 0        n, the number of runs (> kMaxRuns: the rest is not filled)
//   words 1-3     0
//   words 4-19    end[kMaxRuns]
//   words 20-83   bits[kMaxRuns][4]: key c of the tile is bit c%32 of word c/32
constexpr int kMaxRuns = 16;
constexpr int kRunWords = 84;  // 336 bytes, a multiple of 16
// Run table of a virtual key tile (tiling by position): word 0 n, words 4-7 the
// assigned query rows, words 8 + 4r .. 11 + 4r run r = {c0, c1, j0, send}.
constexpr int kVRunWords = 72;  // 288 bytes

// Device image record for one query tile (off_qtile points at an array of these).
struct QTile {
  int32_t row0, row1, ent0, ent1;
};

}  // namespace tree

struct tree_plan {
  tree::Plan p;
};
