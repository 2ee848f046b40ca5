// Host-side plan object shared by the planner (plan.cpp) and the launchers
// (api.cu).  Not part of the public ABI.
#pragma once
#include <vector>

#include "../../include/sp.h"
#include "desc.h"

struct sp_plan {
  sp_shape shape;
  int32_t n_sms = 152;
  int32_t max_pages = 0;
  int32_t n_branches = 0;
  int32_t n_requests = 0;

  // segments, node-token order
  std::vector<int32_t> seg_req, seg_parent, seg_len, seg_round, seg_shared, seg_first_page;
  std::vector<int64_t> seg_node_start;

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

  // device descriptor image (uploaded verbatim)
  std::vector<unsigned char> blob;
  sp::DescHeader hdr{};
  sp_plan_stats stats{};
};
