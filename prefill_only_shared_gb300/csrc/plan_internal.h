// Host-side plan and prefix-cache objects shared by the planner (plan.cpp),
// the cache (cache.cpp) and the launchers (api.cu).  Not part of the public ABI.
#pragma once
#include <utility>
#include <vector>

#include "../../include/sp.h"
#include "desc.h"

// Radix cache of shared segments computed by earlier plans, with the pool
// pages that hold their K/V (LLM2Jev page, section on reusing the radix cache:
// token prefixes whose KV exists are kept across requests and evicted when
// memory is short).  Node 0 is the empty root.
struct sp_cache {
  struct Node {
    std::vector<int32_t> tokens;
    std::vector<int32_t> pages;
    int32_t parent = -1;
    std::vector<int32_t> children;  // in insertion order
    int64_t last_used = 0;
    int32_t pins = 0;  // plans that read the node
    bool alive = true;
  };
  std::vector<Node> nodes;
  std::vector<char> page_free;  // per pool page
  int64_t n_free = 0;
  int64_t clock = 0;
  int64_t evictions = 0;
};

namespace sp {
// Request limits (openjev-sglang article, section on the limits): tokens per
// branch and logical tokens per request.
constexpr int64_t kMaxBranchTokens = 32768;
constexpr int64_t kMaxRequestTokens = 262144;

// Longest cached prefix of seq[0, L): the (node, visible length) chain from
// the root; returns the matched length.
int64_t cache_match(const sp_cache& c, const int32_t* seq, int64_t L,
                    std::vector<std::pair<int32_t, int32_t>>& chain);
// Evict the least recently used unpinned leaf; false when none is evictable.
bool cache_evict_one(sp_cache& c);
// n pages: the lowest run of n free consecutive pages, else the lowest free
// pages (the caller has made sure n pages are free).
void cache_alloc(sp_cache& c, int32_t n, std::vector<int32_t>& out);
}  // namespace sp

struct sp_plan {
  sp_shape shape;
  int32_t n_sms = 152;
  int32_t max_pages = 0;
  int32_t n_branches = 0;
  int32_t n_requests = 0;
  int64_t pool_pages = 0;  // pages of the pool the descriptor may name

  // segments computed by this plan, node-token order
  std::vector<int32_t> seg_req, seg_parent, seg_len, seg_round, seg_shared, seg_first_page;
  std::vector<int64_t> seg_node_start;
  // a branch through each segment and the position of the segment's first
  // token in that branch (row node_start + t is position pos + t of it)
  std::vector<int32_t> seg_branch, seg_pos;

  // branches
  std::vector<int32_t> branch_last_seg, branch_round, branch_recompute;
  std::vector<int64_t> branch_last_row;

  // rounds (CSR)
  std::vector<int32_t> round_off, round_branches;

  // launch lists: calls[kCallKinds * round + kind], kind 0 = prefix (shared
  // segments), 1 = branch (leaves, recomputed rows), 2 = tree (both); round
  // n_rounds = every round at once
  static constexpr int kCallKinds = 3;
  struct Call {
    int64_t append_off = 0, n_append = 0;
    int64_t tile_off = 0, n_tiles = 0;
    int64_t merge_off = 0, n_merges = 0;
    int32_t n_parts = 0;
  };
  std::vector<Call> calls;

  // with a prefix cache: the cache, the nodes this plan reads (pinned until
  // the plan is freed), the match group of each segment and its cached chain
  // end, each new shared segment's tokens and pool pages (owned by the plan
  // until the commit hands them to the cache)
  sp_cache* cache = nullptr;
  std::vector<int32_t> pinned;
  std::vector<int32_t> seg_group;
  std::vector<std::pair<int32_t, int32_t>> group_end;  // (node, visible) or (0, 0)
  std::vector<std::vector<int32_t>> seg_tokens, seg_pages;
  std::vector<int32_t> seg_cache_node;  // inserted node or -1
  bool committed = false;

  // device descriptor image (uploaded verbatim)
  std::vector<unsigned char> blob;
  sp::DescHeader hdr{};
  sp_plan_stats stats{};

  // unpins the cache nodes and returns pages the cache did not take
  ~sp_plan();
};
