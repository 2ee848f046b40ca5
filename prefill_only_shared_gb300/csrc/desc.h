// Device descriptor layout written by the host planner (plan.cpp) and read
// by the attention kernels (attn.cu).  Plain structs, 8-byte aligned.
#pragma once
#include <stdint.h>

namespace sp {

constexpr int kRowsPerTile = 256;  // query rows (token x group-head) per CTA tile: two 128-row halves
constexpr int kKeysPerUnit = 128;  // keys per KV unit (8 pages of 16): one N=128 MMA
constexpr int kPageSize = 16;      // tokens per KV page

// One trie segment.  Its K/V rows are node_start .. node_start + len - 1 of
// the k / v inputs and, once the call that computes it has run and if it is
// shared, pages page_ids[page_off ..] of the pool; its ancestors (root first)
// are chain[chain_off .. chain_off + chain_len).  It is computed in round
// `round`, by the prefix call when `shared` is 1 (an inner trie node: at least
// two branches pass through it), else by the branch call (a leaf, 0).  Shared
// 2 marks a level of the prefix cache: computed by an earlier plan, its
// first `len` keys are read from the pool only.
struct SegDesc {
  int64_t node_start;  // first node-token row
  int32_t len;
  int32_t page_off;
  int32_t chain_off;
  int32_t chain_len;
  int32_t round;
  int32_t shared;
};

// One CTA of attention work: tokens [t0, t0+nt) of segment `seg` (times the
// query heads of one KV head, the innermost part of the launch index), over the KV
// units [u_lo, u_hi) of its context (ancestor units first, then own units up
// to the causal bound).  part < 0: write final out/lse; else write partial
// slot `part`, which the call's merge entry `merge` combines with the other
// parts of the split tile.
// A paired tile (seg2 >= 0) holds the last tokens of two sibling leaves, each
// fitting one 128-row half: half A tokens [t0, t0+nt) of `seg`, half B tokens
// [t0b, t0b+ntb) of `seg2`.  Both read the common ancestors; then come the
// own units of `seg` (half A's) and of `seg2` (half B's), each half masking
// the other's.  Paired tiles are never split.
struct TileDesc {
  int32_t seg, t0, nt, u_lo, u_hi, part;
  int32_t merge, seg2, t0b, ntb;
  int32_t pad0, pad1;
};

// Rows of one split tile whose `nparts` partials start at slot part0.
struct MergeDesc {
  int32_t seg, t0, nt, part0, nparts;
  int32_t pad0, pad1, pad2;
};

// One 16-token page of a shared segment that a call writes into the pool
// (plan metadata: the attention kernel writes the pages of the tiles it runs).
struct AppendDesc {
  int32_t seg, page_in_seg;
};

struct DescHeader {
  int64_t off_segs, off_pages, off_chain, off_append, off_tiles, off_merges;
  int64_t n_segs, n_pages, n_chain, n_append, n_tiles, n_merges;
};

}  // namespace sp
