// Device descriptor layout written by the host planner (plan.cpp) and read
// by the attention kernels (attn.cu).  Plain structs, 8-byte aligned.
#pragma once
#include <stdint.h>

namespace sp {

constexpr int kRowsPerTile = 256;  // query rows (token x group-head) per CTA tile: two 128-row halves
constexpr int kKeysPerUnit = 128;  // keys per KV unit (8 pages of 16): one N=128 MMA
constexpr int kPageSize = 16;      // tokens per KV page

// One trie segment.  Its K/V live in pages page_ids[page_off ..]; its
// ancestors (root first) are chain[chain_off .. chain_off + chain_len).
struct SegDesc {
  int64_t node_start;  // first node-token row
  int32_t len;
  int32_t page_off;
  int32_t chain_off;
  int32_t chain_len;
  int32_t pad0, pad1;
};

// One CTA of attention work: tokens [t0, t0+nt) of segment `seg` (times the
// query heads of one KV head, which is the launch's y index), over the KV
// units [u_lo, u_hi) of its context (ancestor units first, then own units up
// to the causal bound).  part < 0: write final out/lse; else write partial
// slot `part`; the last of the split tile's parts to finish (merge entry
// `merge` of the call) combines them.
struct TileDesc {
  int32_t seg, t0, nt, u_lo, u_hi, part;
  int32_t merge, pad1;
};

// Rows of one split tile whose `nparts` partials start at slot part0.
struct MergeDesc {
  int32_t seg, t0, nt, part0, nparts;
  int32_t pad0, pad1, pad2;
};

// One 16-token page of a segment whose K/V are appended into the pool.
struct AppendDesc {
  int32_t seg, page_in_seg;
};

struct DescHeader {
  int64_t off_segs, off_pages, off_chain, off_append, off_tiles, off_merges;
  int64_t n_segs, n_pages, n_chain, n_append, n_tiles, n_merges;
};

}  // namespace sp
