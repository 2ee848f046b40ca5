// Continuous batching of independent requests: a first-in first-out queue
// and the rule that forms each batch, with one plan per batch.
//
// Sources: openjev-multimodal "performance" page, section on next steps
// (batching across requests to raise throughput), and the SGLang-JAX blog
// translation, section on reducing scheduling overhead (the host prepares
// the next batch while the device computes the current one), prior art.
//
// Rules (the pages leave them open; the oracle states the same ones):
// * a request's size is its node tokens: the positions of its token trie,
//   every distinct prefix of its branches counted once (what its plan
//   computes cold);
// * a batch takes requests from the head of the queue in submission order
//   while its node tokens stay within max_batch_tokens and its request count
//   within max_batch_requests; the first request always goes in, so a
//   request larger than the budget forms a batch of its own;
// * request i of a batch is request id i of the batch's plan, so its node
//   rows follow those of requests 0 .. i-1 (the plan's node-token order).
#include <algorithm>
#include <deque>
#include <new>
#include <vector>

#include "plan_internal.h"

namespace {

using sp::kMaxBranchTokens;
using sp::kMaxRequestTokens;

// Distinct prefixes of a set of sequences: sorted lexicographically, each
// sequence adds its length minus its longest common prefix with the
// sequence before it (the longest with any other sequence up to it).
int64_t node_tokens_of(const std::vector<int64_t>& off, const std::vector<int32_t>& tok) {
  const int32_t n = (int32_t)off.size() - 1;
  std::vector<int32_t> order(n);
  for (int32_t i = 0; i < n; ++i) order[i] = i;
  std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    return std::lexicographical_compare(tok.begin() + off[a], tok.begin() + off[a + 1],
                                        tok.begin() + off[b], tok.begin() + off[b + 1]);
  });
  int64_t total = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = order[i];
    const int64_t len = off[b + 1] - off[b];
    int64_t lcp = 0;
    if (i > 0) {
      const int32_t p = order[i - 1];
      const int64_t lp = off[p + 1] - off[p];
      while (lcp < len && lcp < lp && tok[off[b] + lcp] == tok[off[p] + lcp]) ++lcp;
    }
    total += len - lcp;
  }
  return total;
}

}  // namespace

struct sp_batcher {
  struct Req {
    int64_t id;
    std::vector<int64_t> off;
    std::vector<int32_t> tok;
    int64_t node_tokens;
  };
  sp_shape shape;
  int64_t max_tokens = 0;
  int32_t max_requests = 0;
  std::deque<Req> queue;
  int64_t next_id = 0;
  int64_t queued_tokens = 0;
  // views of the last batch
  std::vector<int64_t> ids;
  std::vector<int32_t> branch_off;
  std::vector<int64_t> row_off;
};

extern "C" sp_status sp_batcher_create(const sp_shape* shape, int64_t max_batch_tokens,
                                       int32_t max_batch_requests, sp_batcher** out) {
  if (!out) return SP_ERR_ARG;
  *out = nullptr;
  if (!shape || max_batch_tokens < 1 || max_batch_requests < 1) return SP_ERR_ARG;
  sp_batcher* b = new (std::nothrow) sp_batcher();
  if (!b) return SP_ERR_ARG;
  b->shape = *shape;
  b->max_tokens = max_batch_tokens;
  b->max_requests = max_batch_requests;
  *out = b;
  return SP_OK;
}

extern "C" void sp_batcher_free(sp_batcher* b) { delete b; }

extern "C" sp_status sp_batcher_submit(sp_batcher* b, int32_t n_branches,
                                       const int64_t* tok_offsets, const int32_t* tokens,
                                       int64_t* out_id, int64_t* out_node_tokens) {
  if (!b || !tok_offsets || !tokens || n_branches < 1 || tok_offsets[0] != 0) return SP_ERR_ARG;
  for (int32_t i = 0; i < n_branches; ++i) {
    const int64_t L = tok_offsets[i + 1] - tok_offsets[i];
    if (L <= 0) return SP_ERR_ARG;
    if (L > kMaxBranchTokens) return SP_ERR_LIMIT;
  }
  if (tok_offsets[n_branches] > kMaxRequestTokens) return SP_ERR_LIMIT;
  sp_batcher::Req r;
  r.id = b->next_id;
  r.off.assign(tok_offsets, tok_offsets + n_branches + 1);
  r.tok.assign(tokens, tokens + tok_offsets[n_branches]);
  r.node_tokens = node_tokens_of(r.off, r.tok);
  if (out_id) *out_id = r.id;
  if (out_node_tokens) *out_node_tokens = r.node_tokens;
  b->queued_tokens += r.node_tokens;
  b->queue.push_back(std::move(r));
  ++b->next_id;
  return SP_OK;
}

extern "C" sp_status sp_batcher_pending(const sp_batcher* b, int32_t* n_requests,
                                        int64_t* n_node_tokens) {
  if (!b) return SP_ERR_ARG;
  if (n_requests) *n_requests = (int32_t)b->queue.size();
  if (n_node_tokens) *n_node_tokens = b->queued_tokens;
  return SP_OK;
}

extern "C" sp_status sp_batcher_next(sp_batcher* b, int32_t max_pages, int32_t n_sms,
                                     sp_plan** out_plan, int32_t* n_requests,
                                     const int64_t** request_ids, const int32_t** branch_off,
                                     const int64_t** row_off) {
  if (!b || !out_plan || !n_requests) return SP_ERR_ARG;
  *out_plan = nullptr;
  *n_requests = 0;
  if (b->queue.empty()) return SP_OK;
  // the batch: the head request, then more while they fit
  int32_t n = 1;
  int64_t tokens = b->queue[0].node_tokens;
  while (n < (int32_t)b->queue.size() && n < b->max_requests &&
         tokens + b->queue[n].node_tokens <= b->max_tokens)
    tokens += b->queue[n++].node_tokens;
  std::vector<int32_t> req;
  std::vector<int64_t> off{0};
  std::vector<int32_t> tok;
  std::vector<int64_t> ids;
  std::vector<int32_t> boff{0};
  std::vector<int64_t> roff{0};
  for (int32_t i = 0; i < n; ++i) {
    const sp_batcher::Req& r = b->queue[i];
    const int32_t nb = (int32_t)r.off.size() - 1;
    for (int32_t j = 0; j < nb; ++j) {
      req.push_back(i);
      off.push_back(off.back() + (r.off[j + 1] - r.off[j]));
    }
    tok.insert(tok.end(), r.tok.begin(), r.tok.end());
    ids.push_back(r.id);
    boff.push_back(boff.back() + nb);
    roff.push_back(roff.back() + r.node_tokens);
  }
  sp_plan* plan = nullptr;
  const sp_status st = sp_plan_build(&b->shape, (int32_t)req.size(), req.data(), off.data(),
                                     tok.data(), max_pages, n_sms, &plan);
  if (st != SP_OK) return st;  // the queue is left as it was
  for (int32_t i = 0; i < n; ++i) {
    b->queued_tokens -= b->queue.front().node_tokens;
    b->queue.pop_front();
  }
  b->ids.swap(ids);
  b->branch_off.swap(boff);
  b->row_off.swap(roff);
  *out_plan = plan;
  *n_requests = n;
  if (request_ids) *request_ids = b->ids.data();
  if (branch_off) *branch_off = b->branch_off.data();
  if (row_off) *row_off = b->row_off.data();
  return SP_OK;
}
